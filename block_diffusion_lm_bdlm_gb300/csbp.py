"""Context-sharded block parallelism (CSBP): the partition of one
[clean | corrupted] sequence over R ranks and the exchange of its clean K/V.

What the pages describe ("Block Parallelism For Efficient Distributed
Long-Context Diffusion Language Model Training", abstract; rit.work CSBP post,
sections on block parallelism and CSBP):
  - block parallelism gives every corrupted target block, with its forward,
    loss and backward, to one rank; its corrupted K/V and their gradients
    never leave that rank;
  - CSBP also shards the shared clean sequence across the ranks, so that no
    rank keeps a replicated clean prefix; only clean K/V and their gradients
    move between ranks;
  - the valid (query, key) pairs are the same as unsharded attention's, and
    early and late blocks are assigned together to balance the work.

The plan (the plainest reading where the pages leave a step open):
  - rank r owns the contiguous clean positions [lo_r, hi_r) (rows and keys);
  - corrupted block p is paired with block nb-1-p, and pair p goes to rank
    p mod R; a rank lists its blocks in ascending order;
  - forward: all-gather the clean K/V shards; each rank then computes its
    clean rows against the clean keys (a key-window call over the rows
    [lo_r, hi_r)) and its corrupted blocks against the clean keys and their
    own corrupted keys (a block-group call); both are complete, so no
    partial merge is needed;
  - backward: each rank takes the same two calls backward, which give the
    complete dq of its rows and the complete dk, dv of its corrupted keys,
    and two shares of the clean keys' dk, dv; the shares of all ranks are
    summed by a reduce-scatter that leaves each clean shard's dk, dv on its
    owner.

The attention itself runs through an `ops` object (GpuOps: the CUDA library;
the tests pass an implementation of the same four calls). The exchange runs
through torch.distributed (NCCL between GPUs; gloo with the tensors staged
through host memory, on CPU or between processes that share a GPU), or, to
emulate all ranks in one process, through run_local.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch


@dataclass(frozen=True)
class RankPlan:
    rank: int
    clean_lo: int               # clean positions [clean_lo, clean_hi) owned by this rank
    clean_hi: int
    blocks: Tuple[int, ...]     # corrupted target blocks owned by this rank, ascending


@dataclass(frozen=True)
class CSBPPlan:
    """The partition of one sequence of clean length n, block size B, over R
    ranks. The clean shards are equal (R must divide n)."""
    n: int
    block: int
    ranks: int
    per_rank: Tuple[RankPlan, ...] = field(repr=False)

    @staticmethod
    def build(n: int, block: int, ranks: int) -> "CSBPPlan":
        if ranks < 1 or n < 1 or block < 1:
            raise ValueError("n, block and ranks must be positive")
        if n % ranks:
            raise ValueError("the clean length must split into equal shards (ranks must divide n)")
        nb = (n + block - 1) // block
        owned: List[List[int]] = [[] for _ in range(ranks)]
        for p in range((nb + 1) // 2):
            r = p % ranks
            owned[r].append(p)
            if nb - 1 - p != p:
                owned[r].append(nb - 1 - p)
        s = n // ranks
        per = tuple(RankPlan(r, r * s, (r + 1) * s, tuple(sorted(owned[r]))) for r in range(ranks))
        return CSBPPlan(n, block, ranks, per)

    def rank(self, r: int) -> RankPlan:
        return self.per_rank[r]

    def corrupted_rows(self, r: int) -> List[int]:
        """Sequence positions (in [n, 2n)) of rank r's corrupted rows, in its
        list order: B per listed block, past the half's end for the padding
        of a short last block (those rows hold no token)."""
        n, B = self.n, self.block
        return [n + b * B + i for b in self.per_rank[r].blocks for i in range(B)]

    def valid_pairs(self, r: int) -> int:
        """Valid (query, key) pairs per head that rank r computes: its clean
        rows against the clean keys they see, its corrupted rows against the
        clean prefix and their own block."""
        n, B = self.n, self.block
        p = self.per_rank[r]
        clean = sum(min(n, (pos // B + 1) * B) for pos in range(p.clean_lo, p.clean_hi))
        corr = 0
        for b in p.blocks:
            rows = min(B, n - b * B)
            corr += rows * (b * B + rows)
        return clean + corr


@dataclass
class RankData:
    """What rank r holds: the rows of its clean shard and of its corrupted
    blocks (q, dO: [rows, H, d]; k, v: [rows, Hk, d]). The corrupted rows
    are laid out as a block group: B rows per listed block, list order."""
    q_clean: torch.Tensor
    k_clean: torch.Tensor
    v_clean: torch.Tensor
    do_clean: torch.Tensor
    q_corr: torch.Tensor
    k_corr: torch.Tensor
    v_corr: torch.Tensor
    do_corr: torch.Tensor
    blocks: torch.Tensor        # int32 block ids (on the compute device)


def split_inputs(plan: CSBPPlan, q, k, v, do, r: int) -> RankData:
    """Rank r's rows of full [2n, ...] tensors (a test and benchmark helper:
    in training each rank produces exactly these rows)."""
    p = plan.rank(r)
    rows = torch.tensor(plan.corrupted_rows(r), dtype=torch.long, device=q.device)
    real = rows < 2 * plan.n
    safe = torch.where(real, rows, torch.zeros_like(rows))

    def corr(t):
        out = t[safe].clone()
        out[~real] = 0  # padding rows of a short last block hold zeros
        return out

    return RankData(q[p.clean_lo:p.clean_hi].contiguous(), k[p.clean_lo:p.clean_hi].contiguous(),
                    v[p.clean_lo:p.clean_hi].contiguous(), do[p.clean_lo:p.clean_hi].contiguous(),
                    corr(q), corr(k), corr(v), corr(do),
                    torch.tensor(p.blocks, dtype=torch.int32, device=q.device))


@dataclass
class RankForward:
    o_clean: torch.Tensor
    lse_clean: torch.Tensor
    o_corr: torch.Tensor
    lse_corr: torch.Tensor


@dataclass
class RankGrads:
    dq_clean: torch.Tensor      # complete, for the rank's clean rows
    dq_corr: torch.Tensor       # complete, for its corrupted rows
    dk_corr: torch.Tensor       # complete, for its corrupted keys
    dv_corr: torch.Tensor
    dk_clean: Optional[torch.Tensor] = None  # after the exchange: complete, for its clean shard
    dv_clean: Optional[torch.Tensor] = None


class GpuOps:
    """The four attention calls of a rank, on the CUDA library."""

    def __init__(self, softmax_scale: float = 0.0):
        import block_diffusion_lm_bdlm_gb300 as bd

        self.bd = bd
        self.scale = softmax_scale

    def fwd_clean(self, q, k_clean, v_clean, n, block, lo, hi):
        bd = self.bd
        return bd.bdlm_attn_fwd(q, k_clean, v_clean, block, L=2 * n, softmax_scale=self.scale,
                                part=bd.Partial.window(0, n, q_lo=lo, q_hi=hi))

    def fwd_group(self, q, k, v, n, block, blocks):
        bd = self.bd
        return bd.bdlm_attn_fwd(q, k, v, block, L=2 * n, softmax_scale=self.scale, part=bd.Partial.group(blocks))

    def bwd_clean(self, q, k_clean, v_clean, o, lse, do, n, block, lo, hi):
        bd = self.bd
        return bd.bdlm_attn_bwd(q, k_clean, v_clean, o, lse, do, block, L=2 * n, softmax_scale=self.scale,
                                part=bd.Partial.window(0, n, q_lo=lo, q_hi=hi))

    def bwd_group(self, q, k, v, o, lse, do, n, block, blocks):
        bd = self.bd
        return bd.bdlm_attn_bwd(q, k, v, o, lse, do, block, L=2 * n, softmax_scale=self.scale,
                                part=bd.Partial.group(blocks))


# ----------------------------------------------------------------------------
# one rank's compute, given the gathered clean K/V
# ----------------------------------------------------------------------------
def rank_forward(plan: CSBPPlan, r: int, x: RankData, k_all, v_all, ops) -> RankForward:
    p = plan.rank(r)
    n, B = plan.n, plan.block
    o_c, l_c = ops.fwd_clean(x.q_clean, k_all, v_all, n, B, p.clean_lo, p.clean_hi)
    if not p.blocks:  # more ranks than block pairs: this rank owns no corrupted block
        H = x.q_corr.shape[1]
        return RankForward(o_c, l_c, torch.empty_like(x.q_corr), l_c.new_empty((H, 0)))
    kg = torch.cat([k_all, x.k_corr])
    vg = torch.cat([v_all, x.v_corr])
    o_g, l_g = ops.fwd_group(x.q_corr, kg, vg, n, B, x.blocks)
    return RankForward(o_c, l_c, o_g, l_g)


def rank_backward(plan: CSBPPlan, r: int, x: RankData, k_all, v_all, f: RankForward, ops):
    """Returns (RankGrads without the clean keys' gradients, the rank's
    shares of the clean keys' dk and dv, [n, Hk, d] each, in fp32 (or the
    inputs' type when wider))."""
    p = plan.rank(r)
    n, B = plan.n, plan.block
    dq_c, dk_c, dv_c = ops.bwd_clean(x.q_clean, k_all, v_all, f.o_clean, f.lse_clean, x.do_clean, n, B,
                                     p.clean_lo, p.clean_hi)
    acc = torch.promote_types(dk_c.dtype, torch.float32)  # the shares add in fp32 (or wider)
    share_k, share_v = dk_c.to(acc), dv_c.to(acc)
    if not p.blocks:
        return RankGrads(dq_c, torch.empty_like(x.q_corr), torch.empty_like(x.k_corr),
                         torch.empty_like(x.v_corr)), share_k, share_v
    kg = torch.cat([k_all, x.k_corr])
    vg = torch.cat([v_all, x.v_corr])
    dq_g, dk_g, dv_g = ops.bwd_group(x.q_corr, kg, vg, f.o_corr, f.lse_corr, x.do_corr, n, B, x.blocks)
    share_k = share_k + dk_g[:n].to(acc)
    share_v = share_v + dv_g[:n].to(acc)
    return RankGrads(dq_c, dq_g, dk_g[n:], dv_g[n:]), share_k, share_v


# ----------------------------------------------------------------------------
# the exchange
# ----------------------------------------------------------------------------
def _staged(t: torch.Tensor, backend: str) -> bool:
    """gloo moves host tensors: device tensors go through host memory."""
    return backend != "nccl" and t.is_cuda


def _gather_clean(t: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of the ranks' clean shards in rank order. Under gloo a
    device tensor is staged through host memory; 16-bit floats travel as
    bytes (an all-gather only copies them, and gloo has no bf16 gather)."""
    import torch.distributed as dist

    backend = dist.get_backend(group)
    src = t.contiguous()
    if _staged(src, backend):
        src = src.cpu()
    wire = src.view(torch.uint8) if src.dtype in (torch.bfloat16, torch.float16) else src
    parts = [torch.empty_like(wire) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, wire, group=group)
    out = torch.cat(parts).view(src.dtype)
    return out.to(t.device) if out.device != t.device else out


def _reduce_scatter_clean(share: torch.Tensor, r: int, ranks: int, group=None) -> torch.Tensor:
    """Sum the ranks' [n, ...] shares and return rows of shard r. NCCL has a
    reduce-scatter; gloo has none, so there the sum is an all-reduce (of a
    host copy when the shares live on a device) and the rank keeps its rows."""
    import torch.distributed as dist

    s = share.shape[0] // ranks
    backend = dist.get_backend(group)
    if backend == "nccl":
        out = torch.empty((s,) + tuple(share.shape[1:]), dtype=share.dtype, device=share.device)
        dist.reduce_scatter_tensor(out, share.contiguous(), op=dist.ReduceOp.SUM, group=group)
        return out
    total = share.cpu() if _staged(share, backend) else share.clone()
    dist.all_reduce(total, op=dist.ReduceOp.SUM, group=group)
    return total[r * s:(r + 1) * s].contiguous().to(share.device)


def run_rank(plan: CSBPPlan, x: RankData, ops, group=None) -> Tuple[RankForward, RankGrads]:
    """Forward and backward of this process's rank under torch.distributed:
    all-gather of the clean K/V, the rank's calls, and the reduce-scatter of
    the clean keys' gradients (results in bf16, as the library's)."""
    import torch.distributed as dist

    r = dist.get_rank(group)
    if dist.get_world_size(group) != plan.ranks:
        raise ValueError("the process group and the plan have different numbers of ranks")
    k_all = _gather_clean(x.k_clean, group)
    v_all = _gather_clean(x.v_clean, group)
    f = rank_forward(plan, r, x, k_all, v_all, ops)
    g, sk, sv = rank_backward(plan, r, x, k_all, v_all, f, ops)
    g.dk_clean = _reduce_scatter_clean(sk, r, plan.ranks, group).to(x.k_clean.dtype)
    g.dv_clean = _reduce_scatter_clean(sv, r, plan.ranks, group).to(x.v_clean.dtype)
    return f, g


def run_local(plan: CSBPPlan, xs: Sequence[RankData], ops) -> List[Tuple[RankForward, RankGrads]]:
    """All ranks in one process (one device): the same calls, with the
    exchange done by concatenation and summation."""
    k_all = torch.cat([x.k_clean for x in xs])
    v_all = torch.cat([x.v_clean for x in xs])
    outs, shares_k, shares_v = [], [], []
    for r, x in enumerate(xs):
        f = rank_forward(plan, r, x, k_all, v_all, ops)
        g, sk, sv = rank_backward(plan, r, x, k_all, v_all, f, ops)
        outs.append((f, g))
        shares_k.append(sk)
        shares_v.append(sv)
    tk = torch.stack(shares_k).sum(0)
    tv = torch.stack(shares_v).sum(0)
    s = plan.n // plan.ranks
    for r, (f, g) in enumerate(outs):
        g.dk_clean = tk[r * s:(r + 1) * s].to(xs[r].k_clean.dtype)
        g.dv_clean = tv[r * s:(r + 1) * s].to(xs[r].v_clean.dtype)
    return outs
