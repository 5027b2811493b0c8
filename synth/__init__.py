"""Seeded synthetic inputs for BDLM attention: shapes, seeds and value
distributions only.

This module holds none of the method's arithmetic (no mask, no softmax, no
merge). It is the one piece shared by the float64 oracle's tests and the CUDA
path's tests and benchmark: both sides receive the same tensors from here.

The five workloads restate the long-context SFT shapes that the paper
"Block Parallelism For Efficient Distributed Long-Context Diffusion Language
Model Training" (abstract) measures on: a [clean | corrupted] concatenation per
sequence, block sizes 16-64, GQA heads and head_dim 128. The models and data of
those runs are not available, so i.i.d. Gaussian tensors of the same shapes
stand in for activations.

Layout (row-major, "thd"): q, o, dO are [L, H, d]; k, v are [Lk, Hk, d];
L counts every row of the concatenation, so one sequence with clean length n
has L = 2n rows (clean rows 0..n-1, then corrupted rows n..2n-1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n: Optional[int]          # clean length of the single sequence (None for packed)
    block: int
    heads: int
    kv_heads: int
    head_dim: int
    seed: int
    qkv_std: float            # q, k, v ~ N(0, qkv_std^2); dO ~ N(0, 1)
    input_fp32: bool = False  # the tiny case is specified in fp32; the GPU path gets bf16(x)
    shards: int = 0           # contiguous clean-K/V shards for the sharded forward + merge
    groups: int = 0           # early/late-paired corrupted-block groups
    docs: int = 0             # packed documents (varlen)
    doc_len_lo: int = 512
    doc_len_hi: int = 32768

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS: List[Workload] = [
    Workload("tiny_n256_b16_h2_d64", n=256, block=16, heads=2, kv_heads=2, head_dim=64,
             seed=0, qkv_std=1.0, input_fp32=True, shards=2),
    Workload("mid_n8192_b32_h32kv8_d128", n=8192, block=32, heads=32, kv_heads=8,
             head_dim=128, seed=1, qkv_std=0.5),
    Workload("long128k_n131072_b64_h32kv8_d128", n=131072, block=64, heads=32, kv_heads=8,
             head_dim=128, seed=2, qkv_std=0.5, shards=8),
    Workload("vlong256k_n262144_b16_h16kv4_d128", n=262144, block=16, heads=16, kv_heads=4,
             head_dim=128, seed=3, qkv_std=0.5, groups=16),
    Workload("packed64_b32_h32kv8_d128", n=None, block=32, heads=32, kv_heads=8,
             head_dim=128, seed=4, qkv_std=0.5, docs=64),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def doc_lengths(w: Workload) -> List[int]:
    """Document lengths (rows, clean + corrupted) of a packed workload.

    u ~ U(0,1) in float64 from a CPU generator seeded with the workload seed;
    length = floor(exp(ln lo + u * ln(hi/lo))) (log-uniform in [lo, hi]),
    rounded down to a multiple of 2*block so that each half holds whole blocks.
    """
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    u = torch.rand(w.docs, generator=g, dtype=torch.float64)
    lo, hi = math.log(w.doc_len_lo), math.log(w.doc_len_hi / w.doc_len_lo)
    lens = []
    for x in u.tolist():
        raw = int(math.floor(math.exp(lo + x * hi)))
        lens.append(max(2 * w.block, (raw // (2 * w.block)) * (2 * w.block)))
    return lens


def cu_seqlens_of(lengths: List[int]) -> List[int]:
    out = [0]
    for x in lengths:
        out.append(out[-1] + x)
    return out


def total_rows(w: Workload) -> int:
    if w.docs:
        return sum(doc_lengths(w))
    return 2 * w.n


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    cu_seqlens: Optional[List[int]] = None
    q_fp32: Optional[torch.Tensor] = field(default=None, repr=False)


def make_inputs(w: Workload, device: str = "cpu", dtype: torch.dtype = torch.bfloat16,
                rows: Optional[int] = None, keep_fp32: bool = False) -> Inputs:
    """Draw q, k, v, dO (in that order) as N(0,1) fp32 from a generator on
    `device` seeded with the workload seed, scale q/k/v by qkv_std, cast to
    `dtype`. `rows` overrides L (used to build small cases of a workload's
    structure). Packed workloads draw their lengths first, on the CPU.
    """
    cu = None
    if w.docs:
        cu = cu_seqlens_of(doc_lengths(w))
        L = cu[-1]
    else:
        L = 2 * w.n if rows is None else rows
    g = torch.Generator(device=device).manual_seed(w.seed)
    shp_q = (L, w.heads, w.head_dim)
    shp_k = (L, w.kv_heads, w.head_dim)

    def draw(shape, std):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x

    q32 = draw(shp_q, w.qkv_std)
    q = q32.to(dtype)
    k = draw(shp_k, w.qkv_std).to(dtype)
    v = draw(shp_k, w.qkv_std).to(dtype)
    do = draw(shp_q, 1.0).to(dtype)
    return Inputs(q=q, k=k, v=v, do=do, cu_seqlens=cu,
                  q_fp32=q32 if keep_fp32 else None)


def shard_bounds(n: int, shards: int) -> List[tuple]:
    """Contiguous clean-key shards [lo, hi) covering clean positions [0, n)."""
    base, rem = divmod(n, shards)
    out, lo = [], 0
    for s in range(shards):
        hi = lo + base + (1 if s < rem else 0)
        out.append((lo, hi))
        lo = hi
    return out


def early_late_groups(n_blocks: int, groups: int) -> List[List[int]]:
    """Corrupted-block groups: block p is paired with block n_blocks-1-p, and
    pair p goes to group p mod groups; each group lists its blocks ascending.
    (An odd middle block, if any, goes to group (n_blocks//2) mod groups.)
    """
    out = [[] for _ in range(groups)]
    for p in range((n_blocks + 1) // 2):
        g = p % groups
        out[g].append(p)
        if n_blocks - 1 - p != p:
            out[g].append(n_blocks - 1 - p)
    return [sorted(x) for x in out]
