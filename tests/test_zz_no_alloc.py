"""bdlm_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory (framework-owned memory, no allocation after start-up).

It is called here through the C ABI with caller-owned outputs only, and its
results are checked against bdlm_attn_fwd (which takes a caller workspace) and
against the float64 oracle on two calls in a row; the second call reuses the
library's fixed scratch that the first one left behind. A call with a bad
block id must report the device check through bdlm_read_error(NULL). The file
is named to run last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import LSE_RTOL, O_ATOL, check_lse, check_o, host

pytestmark = pytest.mark.gpu


def _noalloc(lib, bd, q, k, v, block, o, lse, part=None, L=None):
    Lq, H, d = q.shape
    cpart = ctypes.byref(part.c()) if part is not None else None
    return lib.bdlm_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     Lq if L is None else L, block, H, k.shape[1], d, None, 1, 0.0, cpart,
                                     torch.cuda.current_stream().cuda_stream)


def _close(o, lse, ro, rl):
    assert (o.float() - ro.float()).abs().max().item() <= O_ATOL
    fin = torch.isfinite(rl)
    assert torch.equal(torch.isneginf(lse), torch.isneginf(rl))
    assert ((lse[fin] - rl[fin]).abs() / rl[fin].abs().clamp(min=1.0)).max().item() <= LSE_RTOL


def test_noalloc_forward_matches_the_workspace_forward_twice():
    import block_diffusion_lm_bdlm_gb300 as bd

    lib = bd.load_library()
    # two different calls in a row: a full forward, then a key-window partial
    w = synth.Workload("noalloc", n=1024, block=32, heads=8, kv_heads=2, head_dim=128, seed=21, qkv_std=0.5)
    x = synth.make_inputs(w, device="cuda")
    o = torch.empty_like(x.q)
    lse = torch.empty((w.heads, 2 * w.n), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, bd, x.q, x.k, x.v, w.block, o, lse) == 0
    ro, rl = bd.bdlm_attn_fwd(x.q, x.k, x.v, w.block)
    torch.cuda.synchronize()
    assert bd.bdlm_read_error(None) == 0
    _close(o, lse, ro, rl)
    f64 = lambda t: t.double().cpu().numpy()
    ref = oracle.bdlm_attention(f64(x.q), f64(x.k), f64(x.v), w.block, w.scale)
    check_o(host(o), ref["o"], "noalloc o vs oracle")
    check_lse(host(lse), ref["lse"], "noalloc lse vs oracle")

    lo, hi = 256, 768
    part = bd.Partial.window(lo, hi)
    o2 = torch.empty_like(x.q)
    lse2 = torch.empty_like(lse)
    kw, vw = x.k[lo:hi], x.v[lo:hi]
    assert _noalloc(lib, bd, x.q, kw, vw, w.block, o2, lse2, part=part) == 0
    ro2, rl2 = bd.bdlm_attn_fwd(x.q, kw, vw, w.block, part=part)
    torch.cuda.synchronize()
    assert bd.bdlm_read_error(None) == 0
    _close(o2, lse2, ro2, rl2)
    assert torch.isneginf(rl2).any()  # rows that see nothing of the window
    pref = oracle.partial_attention(f64(x.q), f64(kw), f64(vw), w.n, w.block, lo, hi, w.scale)
    check_o(host(o2), pref["o"], "noalloc window o vs oracle")
    check_lse(host(lse2), pref["lse"], "noalloc window lse vs oracle")


def test_noalloc_reports_device_checks():
    import block_diffusion_lm_bdlm_gb300 as bd

    w = synth.Workload("noalloc_bad", n=256, block=16, heads=4, kv_heads=2, head_dim=64, seed=22, qkv_std=0.5)
    x = synth.make_inputs(w, device="cuda")
    n, B = w.n, w.block
    nb = n // B
    # a block group whose second id is past the last block: the host cannot
    # see device ids, the prologue rejects the list and launches no work
    bad = torch.tensor([0, nb + 3], dtype=torch.int32, device="cuda")
    rows = 2 * B
    q = x.q[n:n + rows].contiguous()
    kv_rows = n + rows
    k, v = x.k[:kv_rows].contiguous(), x.v[:kv_rows].contiguous()
    o, lse = bd.bdlm_attn_fwd_noalloc(q, k, v, B, L=2 * n, part=bd.Partial.group(bad))
    assert bd.bdlm_read_error(None) == 6  # BDLM_ERR_DEVICE_CHECK
    with pytest.raises(bd.BDLMError):
        bd.bdlm_attn_fwd_noalloc(q, k, v, B, L=2 * n, part=bd.Partial.group(bad), check=True)
    # the next good call clears the word again
    good = torch.tensor([0, nb - 1], dtype=torch.int32, device="cuda")
    bd.bdlm_attn_fwd_noalloc(q, k, v, B, L=2 * n, part=bd.Partial.group(good), check=True)
    assert bd.bdlm_read_error(None) == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    import block_diffusion_lm_bdlm_gb300 as bd

    lib = bd.load_library()
    q = torch.zeros(16, 2, 64, dtype=torch.bfloat16, device="cuda")
    L = 1 << 29  # needs far more than the fixed scratch; rejected before any access to q
    assert bd.bdlm_attn_fwd_workspace_bytes(L, 2, 64) > (4 << 20)
    st = lib.bdlm_attn_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), L, 16, 2,
                                   2, 64, None, 1, 0.0, None, None)
    assert st == 3  # BDLM_ERR_WORKSPACE
