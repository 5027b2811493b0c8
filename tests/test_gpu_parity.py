"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs, at sizes the oracle finishes in seconds that still
span several tiles, ragged tails and the degenerate cases of the mask."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check_grad, check_lse, check_o, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    import block_diffusion_lm_bdlm_gb300 as m

    m.load_library()
    return m


def gen(n, block, H, Hk, d, seed, std=0.5, L=None):
    w = synth.Workload("case", n=n, block=block, heads=H, kv_heads=Hk, head_dim=d, seed=seed, qkv_std=std)
    return w, synth.make_inputs(w, device="cuda", rows=L)


def ref_full(x, w, cu=None, heads=None):
    q, k, v, do = host(x.q), host(x.k), host(x.v), host(x.do)
    if heads is not None:
        g0, g1 = heads
        G = w.heads // w.kv_heads
        q, do = q[:, g0 * G:g1 * G], do[:, g0 * G:g1 * G]
        k, v = k[:, g0:g1], v[:, g0:g1]
    return oracle.bdlm_attention(q, k, v, w.block, w.scale, cu_seqlens=cu, do=do)


SHAPES = [
    # n, block, H, Hk, d
    (256, 16, 2, 2, 64),     # the tiny workload's shape
    (96, 16, 4, 1, 128),     # ragged 64-row tiles, GQA 4:1
    (128, 1, 2, 2, 64),      # block = 1: clean half is token-causal
    (128, 128, 2, 1, 128),   # a single block
    (320, 32, 8, 2, 128),    # several tiles per half
    (200, 8, 3, 3, 64),      # odd head count, ragged
    (64, 64, 1, 1, 128),     # one tile of one block
    (40, 8, 2, 1, 64),       # the prefix range's last key tile runs into own-block keys
    (96, 16, 2, 2, 128),     # same, for 128-key tiles
]


@pytest.mark.parametrize("n,block,H,Hk,d", SHAPES)
def test_full_forward_backward(bd, n, block, H, Hk, d):
    w, x = gen(n, block, H, Hk, d, seed=n + block)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block)
    torch.cuda.synchronize()
    r = ref_full(x, w)
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")


def test_tiny_workload_sharded_and_merged(bd):
    w = synth.WORKLOADS[0]
    x = synth.make_inputs(w, device="cuda", keep_fp32=True)
    n = w.n
    r = ref_full(x, w)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, w.block)
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    windows = synth.shard_bounds(n, w.shards) + [(n, 2 * n)]
    parts, lses = [], []
    q64, k64, v64 = host(x.q), host(x.k), host(x.v)
    for lo, hi in windows:
        po, pl = bd.bdlm_attn_fwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), w.block,
                                  part=bd.Partial.window(lo, hi))
        pr = oracle.partial_attention(q64, k64[lo:hi], v64[lo:hi], n, w.block, lo, hi, w.scale)
        check_o(host(po), pr["o"], f"partial[{lo},{hi}) o")
        check_lse(host(pl), pr["lse"], f"partial[{lo},{hi}) lse")
        parts.append(po)
        lses.append(pl)
    mo, ml = bd.bdlm_lse_merge(parts, lses)
    torch.cuda.synchronize()
    check_o(host(mo), r["o"], "merged o")
    check_lse(host(ml), r["lse"], "merged lse")


def test_merge_f32_partials_from_oracle(bd):
    # the merge alone, fed the oracle's own partials (uploaded as fp32)
    n, block, H, Hk, d = 192, 16, 4, 2, 128
    w, x = gen(n, block, H, Hk, d, seed=5)
    q64, k64, v64 = host(x.q), host(x.k), host(x.v)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale)
    windows = synth.shard_bounds(n, 3) + [(n, 2 * n)]
    parts, lses = [], []
    for lo, hi in windows:
        pr = oracle.partial_attention(q64, k64[lo:hi], v64[lo:hi], n, block, lo, hi, w.scale)
        parts.append(torch.from_numpy(pr["o"]).float().cuda())
        lses.append(torch.from_numpy(pr["lse"]).float().cuda())
    mo, ml = bd.bdlm_lse_merge(parts, lses)
    torch.cuda.synchronize()
    check_o(host(mo), full["o"])
    check_lse(host(ml), full["lse"])


def test_merge_edge_cases(bd):
    rows, H, d = 37, 2, 64
    g = torch.Generator(device="cuda").manual_seed(3)
    o1 = torch.randn(rows, H, d, device="cuda", generator=g).to(torch.bfloat16)
    l1 = torch.randn(H, rows, device="cuda", generator=g)
    junk = torch.full((rows, H, d), float("nan"), device="cuda").to(torch.bfloat16)
    ninf = torch.full((H, rows), float("-inf"), device="cuda")
    # single partial: identity
    mo, ml = bd.bdlm_lse_merge([o1], [l1])
    assert torch.equal(mo, o1)
    assert torch.allclose(ml, l1, atol=1e-6)
    # a -inf partial holding NaN is dropped
    mo, ml = bd.bdlm_lse_merge([junk, o1], [ninf, l1])
    assert torch.equal(mo, o1)
    assert torch.allclose(ml, l1, atol=1e-6)
    # all -inf: zeros and -inf
    mo, ml = bd.bdlm_lse_merge([junk, junk], [ninf, ninf])
    assert torch.all(mo == 0) and torch.all(torch.isneginf(ml))
    # equal lse: average, lse + ln 2
    o2 = torch.randn(rows, H, d, device="cuda", generator=g).to(torch.bfloat16)
    mo, ml = bd.bdlm_lse_merge([o1, o2], [l1, l1])
    torch.cuda.synchronize()
    ref = (o1.float() + o2.float()) / 2
    assert (mo.float() - ref).abs().max().item() <= 1e-2
    assert torch.allclose(ml, l1 + math.log(2.0), atol=1e-5)


def test_window_rows_without_keys(bd):
    n, block, H, Hk, d = 256, 32, 2, 1, 128
    w, x = gen(n, block, H, Hk, d, seed=9)
    lo, hi = 192, 256  # a late clean shard: early clean and corrupted rows see nothing of it
    po, pl = bd.bdlm_attn_fwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), block,
                              part=bd.Partial.window(lo, hi))
    torch.cuda.synchronize()
    pr = oracle.partial_attention(host(x.q), host(x.k)[lo:hi], host(x.v)[lo:hi], n, block, lo, hi, w.scale)
    assert np.isneginf(pr["lse"]).sum() > 0
    check_lse(host(pl), pr["lse"])
    check_o(host(po), pr["o"])
    empty = np.isneginf(pr["lse"]).T
    assert np.all(host(po)[empty] == 0.0)


@pytest.mark.parametrize("n,block,H,Hk,groups", [(512, 16, 4, 2, 4), (384, 32, 2, 1, 3)])
def test_block_groups(bd, n, block, H, Hk, groups):
    d = 128
    w, x = gen(n, block, H, Hk, d, seed=11)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    q64, k64, v64 = host(x.q), host(x.k), host(x.v)
    for blocks in synth.early_late_groups(n // block, groups):
        qpos, kpos = oracle.group_positions(n, block, blocks)
        qi = torch.from_numpy(qpos).cuda()
        ki = torch.from_numpy(kpos).cuda()
        bl = torch.tensor(blocks, dtype=torch.int32, device="cuda")
        go, gl = bd.bdlm_attn_fwd(x.q[qi].contiguous(), x.k[ki].contiguous(), x.v[ki].contiguous(), block,
                                  L=2 * n, part=bd.Partial.group(bl))
        torch.cuda.synchronize()
        r = oracle.group_attention(q64[qpos], k64[kpos], v64[kpos], n, block, blocks, w.scale)
        check_o(host(go), r["o"], "group o")
        check_lse(host(gl), r["lse"], "group lse")
        # equal to the unsplit call on the same rows
        assert (go.float() - o[qi].float()).abs().max().item() <= 2e-2
        assert (gl - lse[:, qi]).abs().max().item() <= 1e-3 * max(1.0, lse.abs().max().item())


# running merge: each window merged into (o, lse) in the forward's epilogue
@pytest.mark.parametrize("n,block,H,Hk,d,shards", [(256, 16, 2, 2, 64, 2), (320, 32, 8, 2, 128, 3),
                                                   (96, 16, 4, 1, 128, 8)])
@pytest.mark.parametrize("o_dtype", [torch.bfloat16, torch.float32])
def test_running_merge_in_forward(bd, n, block, H, Hk, d, shards, o_dtype):
    w, x = gen(n, block, H, Hk, d, seed=5 * n + shards)
    full = oracle.bdlm_attention(host(x.q), host(x.k), host(x.v), block, w.scale)
    windows = synth.shard_bounds(n, shards) + [(n, 2 * n)]
    o = torch.empty(x.q.shape, dtype=o_dtype, device="cuda")
    lse = torch.empty((H, 2 * n), dtype=torch.float32, device="cuda")
    ws = torch.empty(bd.bdlm_attn_fwd_workspace_bytes(2 * n, H, d, 1), dtype=torch.uint8, device="cuda")
    for i, (lo, hi) in enumerate(windows):
        prev_o, prev_l = o.clone(), lse.clone()
        bd.bdlm_attn_fwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), block,
                         part=bd.Partial.window(lo, hi, accumulate=i > 0), out=o, lse=lse, workspace=ws)
        assert bd.bdlm_read_error(ws) == 0
        if i > 0:
            # rows that see no key of this window keep their running result bit for bit
            pr = oracle.partial_attention(host(x.q), host(x.k)[lo:hi], host(x.v)[lo:hi], n, block, lo, hi, w.scale)
            unseen = torch.from_numpy(np.isneginf(pr["lse"])).cuda()
            assert torch.equal(lse[unseen], prev_l[unseen])
            assert torch.equal(o.transpose(0, 1)[unseen], prev_o.transpose(0, 1)[unseen])
    torch.cuda.synchronize()
    check_o(host(o), full["o"], "running-merge o")
    check_lse(host(lse), full["lse"], "running-merge lse")


# sharded backward: each clean-K/V shard (and the local corrupted keys) with
# the merged forward's o and lse; shares of dq sum to the full dq
SHARDED = [
    # n, block, H, Hk, d, shards
    (256, 16, 2, 2, 64, 2),    # the tiny workload's shape and split (d 64)
    (320, 32, 8, 2, 128, 3),   # uneven shards, not block-aligned
    (96, 16, 4, 1, 128, 8),    # windows shorter than one block
    (200, 8, 3, 3, 64, 3),     # odd heads, ragged
]


@pytest.mark.parametrize("n,block,H,Hk,d,shards", SHARDED)
def test_sharded_backward(bd, n, block, H, Hk, d, shards):
    w, x = gen(n, block, H, Hk, d, seed=3 * n + shards)
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, do=do64)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    ws = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(2 * n, H, d, 1), dtype=torch.uint8, device="cuda")
    dq_sum = torch.zeros(2 * n, H, d, dtype=torch.float32, device="cuda")
    dk_cat, dv_cat = torch.empty_like(x.k), torch.empty_like(x.v)
    for lo, hi in synth.shard_bounds(n, shards) + [(n, 2 * n)]:
        dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), o, lse, x.do, block,
                                      part=bd.Partial.window(lo, hi), workspace=ws)
        assert bd.bdlm_read_error(ws) == 0
        r = oracle.partial_attention(q64, k64[lo:hi], v64[lo:hi], n, block, lo, hi, w.scale, do=do64,
                                     o_full=full["o"], lse_full=full["lse"])
        check_grad(host(dq), r["dq"], f"dq share [{lo},{hi})")
        check_grad(host(dk), r["dk"], f"dk [{lo},{hi})")
        check_grad(host(dv), r["dv"], f"dv [{lo},{hi})")
        dq_sum += dq.float()
        dk_cat[lo:hi] = dk
        dv_cat[lo:hi] = dv
    torch.cuda.synchronize()
    check_grad(host(dq_sum), full["dq"], "sum of dq shares")
    check_grad(host(dk_cat), full["dk"], "dk over all shards")
    check_grad(host(dv_cat), full["dv"], "dv over all shards")


@pytest.mark.parametrize("n,block,H,Hk,d,groups", [(512, 16, 4, 2, 128, 4), (384, 32, 2, 1, 128, 3),
                                                   (256, 16, 2, 2, 64, 3)])
def test_block_group_backward(bd, n, block, H, Hk, d, groups):
    w, x = gen(n, block, H, Hk, d, seed=13 + n)
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    dq_full, dk_full, dv_full = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block)
    ws = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(2 * n, H, d, 1), dtype=torch.uint8, device="cuda")
    nb = n // block
    # the early/late groups, plus a group of early blocks only: clean keys
    # from its last block on are seen by none of its rows (zero gradient)
    lists = synth.early_late_groups(nb, groups) + [[0, 2]]
    for blocks in lists:
        qpos, kpos = oracle.group_positions(n, block, blocks)
        qi, ki = torch.from_numpy(qpos).cuda(), torch.from_numpy(kpos).cuda()
        bl = torch.tensor(blocks, dtype=torch.int32, device="cuda")
        part = bd.Partial.group(bl)
        qg, kg, vg, dog = (t[i].contiguous() for t, i in ((x.q, qi), (x.k, ki), (x.v, ki), (x.do, qi)))
        go, gl = bd.bdlm_attn_fwd(qg, kg, vg, block, L=2 * n, part=part)
        dq, dk, dv = bd.bdlm_attn_bwd(qg, kg, vg, go, gl, dog, block, L=2 * n, part=part, workspace=ws)
        assert bd.bdlm_read_error(ws) == 0
        r = oracle.group_attention(q64[qpos], k64[kpos], v64[kpos], n, block, blocks, w.scale, do=do64[qpos])
        check_grad(host(dq), r["dq"], f"group {blocks[:2]} dq")
        check_grad(host(dk), r["dk"], f"group {blocks[:2]} dk")
        check_grad(host(dv), r["dv"], f"group {blocks[:2]} dv")
        # dq of the group's rows and dk, dv of its corrupted keys are complete
        corr = slice(n, None)
        assert (dq.float() - dq_full[qi].float()).norm() <= 1e-2 * dq_full[qi].float().norm()
        assert (dk[corr].float() - dk_full[qi].float()).norm() <= 1e-2 * dk_full[qi].float().norm()
        assert (dv[corr].float() - dv_full[qi].float()).norm() <= 1e-2 * dv_full[qi].float().norm()
        unseen = max(blocks) * block
        assert torch.all(dk[unseen:n] == 0) and torch.all(dv[unseen:n] == 0)


def test_block_group_backward_needs_ascending_blocks(bd):
    n, block, H, Hk, d = 128, 16, 2, 1, 128
    w, x = gen(n, block, H, Hk, d, seed=17)
    blocks = [5, 1]
    qpos, kpos = oracle.group_positions(n, block, blocks)
    qi, ki = torch.from_numpy(qpos).cuda(), torch.from_numpy(kpos).cuda()
    part = bd.Partial.group(torch.tensor(blocks, dtype=torch.int32, device="cuda"))
    qg, kg, vg, dog = (t[i].contiguous() for t, i in ((x.q, qi), (x.k, ki), (x.v, ki), (x.do, qi)))
    go, gl = bd.bdlm_attn_fwd(qg, kg, vg, block, L=2 * n, part=part)  # the forward takes any order
    ws = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(2 * n, H, d, 1), dtype=torch.uint8, device="cuda")
    bd.bdlm_attn_bwd(qg, kg, vg, go, gl, dog, block, L=2 * n, part=part, workspace=ws)
    assert bd.bdlm_read_error(ws) == 6  # BDLM_ERR_DEVICE_CHECK


def test_packed_documents(bd):
    block, H, Hk, d = 32, 4, 2, 128
    lens = [128, 64, 320, 192, 64]
    cu = synth.cu_seqlens_of(lens)
    g = torch.Generator(device="cuda").manual_seed(13)
    T = cu[-1]
    mk = lambda *s: (torch.randn(*s, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    q, k, v = mk(T, H, d), mk(T, Hk, d), mk(T, Hk, d)
    do = (torch.randn(T, H, d, device="cuda", generator=g)).to(torch.bfloat16)
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o, lse = bd.bdlm_attn_fwd(q, k, v, block, cu_seqlens=cu_d)
    dq, dk, dv = bd.bdlm_attn_bwd(q, k, v, o, lse, do, block, cu_seqlens=cu_d)
    torch.cuda.synchronize()
    r = oracle.bdlm_attention(host(q), host(k), host(v), block, 1 / math.sqrt(d), cu_seqlens=cu, do=host(do))
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")


# token-level tasks: (query row range) x (key window) over one sequence
@pytest.mark.parametrize("n,block,H,Hk,d", [(100, 16, 4, 2, 128), (90, 8, 2, 2, 64)])
def test_row_range_by_key_window_tasks(bd, n, block, H, Hk, d):
    w, x = gen(n, block, H, Hk, d, seed=23 + n)
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, do=do64)
    o_g, lse_g = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)  # the backward's softmax statistics
    row_cuts = [0, 7, n - 3, n, n + 13, 2 * n]
    key_cuts = [0, 11, n - 5, n, n + 20, 2 * n]
    L = 2 * n
    dk = torch.zeros(x.k.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros(x.v.shape, dtype=torch.float32, device="cuda")
    for qa, qb in zip(row_cuts[:-1], row_cuts[1:]):
        qr, dor = x.q[qa:qb].contiguous(), x.do[qa:qb].contiguous()
        o = torch.empty(qr.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty((H, qb - qa), dtype=torch.float32, device="cuda")
        dq = torch.zeros(qr.shape, dtype=torch.float32, device="cuda")
        for i, (ka, kb) in enumerate(zip(key_cuts[:-1], key_cuts[1:])):
            kw, vw = x.k[ka:kb].contiguous(), x.v[ka:kb].contiguous()
            bd.bdlm_attn_fwd(qr, kw, vw, block, L=L, out=o, lse=lse,
                             part=bd.Partial.window(ka, kb, accumulate=i > 0, q_lo=qa, q_hi=qb))
            sq, sk, sv = bd.bdlm_attn_bwd(qr, kw, vw, o_g[qa:qb].contiguous(), lse_g[:, qa:qb].contiguous(), dor,
                                          block, L=L, part=bd.Partial.window(ka, kb, q_lo=qa, q_hi=qb))
            dq += sq.float()
            dk[ka:kb] += sk.float()
            dv[ka:kb] += sv.float()
        torch.cuda.synchronize()
        check_o(host(o), full["o"][qa:qb], f"rows [{qa},{qb}) o")
        check_lse(host(lse), full["lse"][:, qa:qb], f"rows [{qa},{qb}) lse")
        check_grad(host(dq), full["dq"][qa:qb], f"rows [{qa},{qb}) dq")
    check_grad(host(dk), full["dk"], "dk over all tasks")
    check_grad(host(dv), full["dv"], "dv over all tasks")


# ragged last blocks: B does not divide the clean length
RAGGED = [
    # n, block, H, Hk, d
    (100, 16, 2, 1, 128),   # 6 whole blocks + 4 rows
    (70, 32, 4, 2, 64),     # d 64 backward
    (45, 8, 3, 3, 128),
    (37, 64, 2, 2, 128),    # B > n: one short block per half
    (129, 128, 2, 1, 128),  # one whole block and one row
    (300, 64, 4, 1, 128),   # several 128-row tiles, short last block
    (300, 200, 2, 1, 128),  # blocks longer than a 128-row tile, short last block
]


@pytest.mark.parametrize("n,block,H,Hk,d", RAGGED)
def test_ragged_last_block(bd, n, block, H, Hk, d):
    w, x = gen(n, block, H, Hk, d, seed=7 * n + block)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block)
    torch.cuda.synchronize()
    r = ref_full(x, w)
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")


def test_ragged_packed_documents(bd):
    block, H, Hk, d = 16, 4, 2, 128
    lens = [2 * 37, 2 * 100, 2 * 5, 2 * 129, 2 * 64, 2 * 1]
    cu = synth.cu_seqlens_of(lens)
    g = torch.Generator(device="cuda").manual_seed(17)
    T = cu[-1]
    mk = lambda *s: (torch.randn(*s, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    q, k, v = mk(T, H, d), mk(T, Hk, d), mk(T, Hk, d)
    do = (torch.randn(T, H, d, device="cuda", generator=g)).to(torch.bfloat16)
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o, lse = bd.bdlm_attn_fwd(q, k, v, block, cu_seqlens=cu_d)
    dq, dk, dv = bd.bdlm_attn_bwd(q, k, v, o, lse, do, block, cu_seqlens=cu_d)
    torch.cuda.synchronize()
    r = oracle.bdlm_attention(host(q), host(k), host(v), block, 1 / math.sqrt(d), cu_seqlens=cu, do=host(do))
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")


def test_ragged_sharded_forward_merge_backward(bd):
    n, block, H, Hk, d = 100, 16, 4, 2, 128
    w, x = gen(n, block, H, Hk, d, seed=19)
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, do=do64)
    windows = synth.shard_bounds(n, 3) + [(n, 2 * n)]
    parts, lses = [], []
    for lo, hi in windows:
        po, pl = bd.bdlm_attn_fwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), block,
                                  part=bd.Partial.window(lo, hi))
        parts.append(po)
        lses.append(pl)
    o, lse = bd.bdlm_lse_merge(parts, lses)
    dq_sum = torch.zeros(x.q.shape, dtype=torch.float32, device="cuda")
    dk, dv = torch.empty_like(x.k), torch.empty_like(x.v)
    for lo, hi in windows:
        sq, sk, sv = bd.bdlm_attn_bwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), o, lse, x.do, block,
                                      part=bd.Partial.window(lo, hi))
        dq_sum += sq.float()
        dk[lo:hi] = sk
        dv[lo:hi] = sv
    torch.cuda.synchronize()
    check_o(host(o), full["o"], "merged o")
    check_lse(host(lse), full["lse"], "merged lse")
    check_grad(host(dq_sum), full["dq"], "sum of dq shares")
    check_grad(host(dk), full["dk"], "dk")
    check_grad(host(dv), full["dv"], "dv")


def test_zero_keys_closed_form(bd):
    n, block, H, d = 192, 16, 2, 128
    w, x = gen(n, block, H, H, d, seed=17)
    k = torch.zeros_like(x.k)
    o, lse = bd.bdlm_attn_fwd(x.q, k, x.v, block)
    torch.cuda.synchronize()
    lse_h = host(lse)
    v = host(x.v)
    o_h = host(o)
    for i in range(2 * n):
        b = (i % n) // block
        assert np.all(np.abs(lse_h[:, i] - math.log((b + 1) * block)) <= 1e-5 * math.log((b + 1) * block) + 1e-6)
        vis = np.arange(0, (b + 1) * block) if i < n else np.concatenate(
            [np.arange(0, b * block), n + b * block + np.arange(block)])
        assert np.abs(o_h[i] - v[vis].mean(axis=0)).max() <= 8e-3


def test_malformed_cu_seqlens_is_reported(bd):
    block, H, d = 32, 2, 64
    T = 256
    q = torch.zeros(T, H, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bd.bdlm_attn_fwd_workspace_bytes(T, H, d, 2), dtype=torch.uint8, device="cuda")
    # odd document length, an empty document, decreasing offsets, wrong total
    for bad in ([0, 63, 256], [0, 0, 256], [0, 200, 128], [0, 128, 200]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        bd.bdlm_attn_fwd(q, q, q, block, cu_seqlens=cu, workspace=ws)
        assert bd.bdlm_read_error(ws) == 6, bad
    for good in ([0, 128, 256], [0, 96, 256]):  # the second has short last blocks (48 and 80 clean rows, B = 32)
        cu = torch.tensor(good, dtype=torch.int32, device="cuda")
        bd.bdlm_attn_fwd(q, q, q, block, cu_seqlens=cu, workspace=ws)
        assert bd.bdlm_read_error(ws) == 0, good


def test_forward_is_deterministic(bd):
    w, x = gen(512, 32, 4, 2, 128, seed=19)
    o1, l1 = bd.bdlm_attn_fwd(x.q, x.k, x.v, 32)
    o2, l2 = bd.bdlm_attn_fwd(x.q, x.k, x.v, 32)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mid_workload(bd):
    """8192 + 8192 rows, 32/8 heads, B = 32: one kv group in full (o, lse, all
    gradients) and 8 sampled query blocks on every head (o, lse, dq)."""
    w = synth.WORKLOADS[1]
    x = synth.make_inputs(w, device="cuda")
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, w.block)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, w.block)
    torch.cuda.synchronize()
    G = w.heads // w.kv_heads
    r = ref_full(x, w, heads=(0, 1))
    check_o(host(o[:, :G]), r["o"])
    check_lse(host(lse[:G]), r["lse"])
    check_grad(host(dq[:, :G]), r["dq"], "dq")
    check_grad(host(dk[:, :1]), r["dk"], "dk")
    check_grad(host(dv[:, :1]), r["dv"], "dv")
    n, B = w.n, w.block
    nb = n // B
    picks = [0, nb // 3, nb - 1]
    blocks = [(0, b * B) for b in picks] + [(0, n + b * B) for b in picks + [nb // 2, 1]]
    rows = np.concatenate([np.arange(r0, r0 + B) for _, r0 in blocks])
    rs = oracle.bdlm_attention(host(x.q), host(x.k), host(x.v), B, w.scale, do=host(x.do), row_blocks=blocks,
                               want_kv_grads=False)
    check_o(host(o)[rows], rs["o"][rows], "sampled o")
    check_lse(host(lse)[:, rows], rs["lse"][:, rows], "sampled lse")
    check_grad(host(dq)[rows], rs["dq"][rows], "sampled dq")


# token-level task lists: one launch over tasks of several packed sequences
TASK_CASES = [
    # sequence clean lengths, block, H, Hk, d, o dtype
    ((300, 200), 32, 4, 2, 128, torch.bfloat16),
    ((300, 200), 32, 4, 2, 128, torch.float32),
    ((129, 70, 256), 48, 2, 1, 128, torch.bfloat16),  # B divides none of them
    ((150, 64), 16, 4, 4, 64, torch.float32),
]


def _task_grid(bd, starts, ns, rng):
    """Per sequence: its rows cut into 3 ranges and its keys into 3 windows;
    task (range, window w) writes slot w. Plus one task per sequence into
    slot 3 on a random row range and key window."""
    tasks = []
    for s0, n in zip(starts, ns):
        rc = [0, int(rng.integers(1, n)), int(rng.integers(n, 2 * n)), 2 * n]
        kc = [0, int(rng.integers(1, n)), int(rng.integers(n, 2 * n)), 2 * n]
        for qa, qb in zip(rc[:-1], rc[1:]):
            for w, (ka, kb) in enumerate(zip(kc[:-1], kc[1:])):
                tasks.append(bd.Task(s0, n, qa, qb, ka, kb, w))
        qa = int(rng.integers(0, 2 * n - 1))
        ka = int(rng.integers(0, 2 * n - 1))
        tasks.append(bd.Task(s0, n, qa, int(rng.integers(qa + 1, 2 * n + 1)), ka, int(rng.integers(ka + 1, 2 * n + 1)), 3))
    rng.shuffle(tasks)
    return tasks


@pytest.mark.parametrize("ns,block,H,Hk,d,odt", TASK_CASES)
def test_task_list_forward(bd, ns, block, H, Hk, d, odt):
    L = 2 * sum(ns)
    starts = [int(s) for s in np.cumsum([0] + [2 * n for n in ns[:-1]])]
    w, x = gen(ns[0], block, H, Hk, d, seed=31 + L, L=L)
    tasks = _task_grid(bd, starts, ns, np.random.default_rng(L))
    S = 4
    # sentinels in the rows no task of a slot covers must survive
    o = torch.full((S, L, H, d), 7.0, dtype=odt, device="cuda")
    lse = torch.full((S, H, L), 3.0, dtype=torch.float32, device="cuda")
    bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, block, tasks, S, out=o, lse=lse)
    torch.cuda.synchronize()
    ref = [dict(seq_start=t.seq_start, n=t.n, q_lo=t.q_lo, q_hi=t.q_hi, key_lo=t.key_lo, key_hi=t.key_hi,
                slot=t.slot) for t in tasks]
    ro, rl = oracle.task_attention(host(x.q), host(x.k), host(x.v), block, w.scale, ref, S)
    go, gl = host(o), host(lse)
    for s in range(S):
        cov = ~np.isnan(rl[s, 0])
        check_o(go[s][cov], ro[s][cov], f"slot {s} o")
        check_lse(gl[s][:, cov], rl[s][:, cov], f"slot {s} lse")
        assert np.all(go[s][~cov] == 7.0) and np.all(gl[s][:, ~cov] == 3.0), f"slot {s}: uncovered rows written"
    # the slots 0-2 of each row split its keys: merged, they give the sequence's attention
    om, lm = bd.bdlm_lse_merge([o[s] for s in range(3)], [lse[s] for s in range(3)])
    torch.cuda.synchronize()
    full = oracle.bdlm_attention(host(x.q), host(x.k), host(x.v), block, w.scale,
                                 cu_seqlens=np.array(starts + [L], dtype=np.int64))
    check_o(host(om), full["o"], "merged o")
    check_lse(host(lm), full["lse"], "merged lse")


def test_task_list_equals_window_calls(bd):
    # the 8 clean shards + local corrupted keys of one sequence as one task
    # list give the same bits as 9 key-window calls (same tiles, same order
    # of arithmetic within a tile)
    n, block, H, Hk, d = 1024, 32, 8, 2, 128
    w, x = gen(n, block, H, Hk, d, seed=77)
    cuts = [i * n // 8 for i in range(9)] + [2 * n]
    tasks = [bd.Task(0, n, 0, 2 * n, a, b, i) for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:]))]
    o, lse = bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, block, tasks, len(tasks))
    assert bd.bdlm_last_launch_count() == 3  # upload, prologue, attention
    for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        ow, lw = bd.bdlm_attn_fwd(x.q, x.k[a:b].contiguous(), x.v[a:b].contiguous(), block,
                                  part=bd.Partial.window(a, b))
        torch.cuda.synchronize()
        assert torch.equal(o[i], ow), f"window {i}: o differs"
        assert torch.equal(lse[i], lw), f"window {i}: lse differs"


def test_task_list_rows_that_see_no_key(bd):
    # clean rows against corrupted keys: o = 0, lse = -inf
    n, block, H, Hk, d = 200, 16, 2, 1, 128
    w, x = gen(n, block, H, Hk, d, seed=78)
    o, lse = bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, block, [bd.Task(0, n, 0, n, n, 2 * n, 0)], 1,
                                    out=torch.full((1, 2 * n, H, d), 5.0, dtype=torch.bfloat16, device="cuda"),
                                    lse=torch.full((1, H, 2 * n), 5.0, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(o[0, :n] == 0) and torch.all(torch.isneginf(lse[0, :, :n]))
    assert torch.all(o[0, n:] == 5.0) and torch.all(lse[0, :, n:] == 5.0)


TASK_BWD_CASES = [
    # sequence clean lengths, block, H, Hk, d
    ((300, 200), 32, 4, 2, 128),
    ((129, 70, 256), 48, 2, 1, 128),  # B divides none of them
    ((150, 64), 16, 4, 4, 64),        # d 64 backward
]


@pytest.mark.parametrize("ns,block,H,Hk,d", TASK_BWD_CASES)
def test_task_list_backward(bd, ns, block, H, Hk, d):
    # per sequence: rows cut into 3 ranges (slot = range), keys into 3
    # windows; plus slot 3 holding one task per sequence on part of its keys
    L = 2 * sum(ns)
    starts = [int(s) for s in np.cumsum([0] + [2 * n for n in ns[:-1]])]
    w, x = gen(ns[0], block, H, Hk, d, seed=41 + L, L=L)
    rng = np.random.default_rng(L + 1)
    tasks = []
    for s0, n in zip(starts, ns):
        rc = [0, int(rng.integers(1, n)), int(rng.integers(n, 2 * n)), 2 * n]
        kc = [0, int(rng.integers(1, n)), int(rng.integers(n, 2 * n)), 2 * n]
        for r, (qa, qb) in enumerate(zip(rc[:-1], rc[1:])):
            for ka, kb in zip(kc[:-1], kc[1:]):
                tasks.append(bd.Task(s0, n, qa, qb, ka, kb, r))
        ka = int(rng.integers(0, 2 * n - 1))
        tasks.append(bd.Task(s0, n, 0, 2 * n, ka, int(rng.integers(ka + 1, 2 * n + 1)), 3))
    rng.shuffle(tasks)
    S = 4
    cu = torch.tensor(starts + [L], dtype=torch.int32, device="cuda")
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block, cu_seqlens=cu)  # the full softmax of every row
    dk = torch.full((S, L, Hk, d), 7.0, dtype=torch.bfloat16, device="cuda")
    dv = torch.full((S, L, Hk, d), 7.0, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = bd.bdlm_attn_bwd_tasks(x.q, x.k, x.v, o, lse, x.do, block, tasks, S, dk=dk, dv=dv)
    torch.cuda.synchronize()
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, cu_seqlens=np.array(starts + [L]), do=do64)
    ref = [dict(seq_start=t.seq_start, n=t.n, q_lo=t.q_lo, q_hi=t.q_hi, key_lo=t.key_lo, key_hi=t.key_hi,
                slot=t.slot) for t in tasks]
    rq, rk, rv = oracle.task_attention_bwd(q64, k64, v64, full["o"], full["lse"], do64, block, w.scale, ref, S)
    check_grad(host(dq), rq, "dq (sum over the tasks)")
    gk, gv = host(dk), host(dv)
    for s in range(S):
        cov = ~np.isnan(rk[s, :, 0, 0])
        check_grad(gk[s][cov], rk[s][cov], f"slot {s} dk")
        check_grad(gv[s][cov], rv[s][cov], f"slot {s} dv")
        assert np.all(gk[s][~cov] == 7.0) and np.all(gv[s][~cov] == 7.0), f"slot {s}: uncovered keys written"
    # slots 0-2 partition every sequence's rows x keys: their sum is the full gradient
    check_grad(gk[:3].sum(axis=0), full["dk"], "dk summed over the row-range slots")
    check_grad(gv[:3].sum(axis=0), full["dv"], "dv summed over the row-range slots")


def test_task_list_with_many_tasks(bd):
    # 1200 one-row tasks: more than one upload launch (960 records each) and
    # more than one enumeration chunk (1024 tasks each), forward and backward
    ns = (120, 80)
    block, H, Hk, d = 16, 2, 1, 128
    L = 2 * sum(ns)
    starts = [0, 2 * ns[0]]
    w, x = gen(ns[0], block, H, Hk, d, seed=97, L=L)
    fwd_tasks, bwd_tasks = [], []
    slot = 0
    for s0, n in zip(starts, ns):
        kc = [0, n // 2, n + 5, 2 * n]
        for p in range(2 * n):
            for wi, (ka, kb) in enumerate(zip(kc[:-1], kc[1:])):
                fwd_tasks.append(bd.Task(s0, n, p, p + 1, ka, kb, wi))
                bwd_tasks.append(bd.Task(s0, n, p, p + 1, ka, kb, slot))
            slot += 1
    assert len(fwd_tasks) == 1200
    o, lse = bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, block, fwd_tasks, 3)
    assert bd.bdlm_last_launch_count() == 4  # two uploads, prologue, attention
    cu = torch.tensor(starts + [L], dtype=torch.int32, device="cuda")
    fo, fl = bd.bdlm_attn_fwd(x.q, x.k, x.v, block, cu_seqlens=cu)
    dq, dk, dv = bd.bdlm_attn_bwd_tasks(x.q, x.k, x.v, fo, fl, x.do, block, bwd_tasks, slot)
    torch.cuda.synchronize()
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    ref = lambda ts: [dict(seq_start=t.seq_start, n=t.n, q_lo=t.q_lo, q_hi=t.q_hi, key_lo=t.key_lo,
                           key_hi=t.key_hi, slot=t.slot) for t in ts]
    ro, rl = oracle.task_attention(q64, k64, v64, block, w.scale, ref(fwd_tasks), 3)
    for s in range(3):
        check_o(host(o[s]), ro[s], f"slot {s} o")
        check_lse(host(lse[s]), rl[s], f"slot {s} lse")
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, cu_seqlens=np.array(starts + [L]), do=do64)
    rq, rk, rv = oracle.task_attention_bwd(q64, k64, v64, full["o"], full["lse"], do64, block, w.scale,
                                           ref(bwd_tasks), slot)
    check_grad(host(dq), rq, "dq")
    # each slot holds one row's contribution to its sequence's keys: compare the
    # sums over the slots (the full gradients) and every slot's covered keys
    gk, gv = host(dk), host(dv)
    check_grad(gk.sum(axis=0), full["dk"], "dk over all slots")
    check_grad(gv.sum(axis=0), full["dv"], "dv over all slots")
    cov = ~np.isnan(rk[:, :, 0, 0])
    err = np.abs(gk[cov] - rk[cov]).max()
    assert err <= 2e-2, f"per-slot dk max abs err {err:.3e}"


def test_step_captured_in_a_cuda_graph(bd):
    # the library's compute calls only launch kernels on the given stream
    # (kernel parameters carry every host-side value), so a whole step can be
    # captured once and replayed on new inputs copied into the same buffers
    n, block, H, Hk, d = 512, 32, 4, 2, 128
    w, x = gen(n, block, H, Hk, d, seed=99)
    L = 2 * n
    wins = [(0, n // 2), (n // 2, n), (n, 2 * n)]
    parts = [torch.empty_like(x.q) for _ in wins]
    plse = [torch.empty((H, L), dtype=torch.float32, device="cuda") for _ in wins]
    o = torch.empty_like(x.q)
    lse = torch.empty((H, L), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(x.q), torch.empty_like(x.k), torch.empty_like(x.v)
    wsf = torch.empty(bd.bdlm_attn_fwd_workspace_bytes(L, H, d), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(L, H, d), dtype=torch.uint8, device="cuda")
    tasks = [bd.Task(0, n, 0, L, lo, hi, i) for i, (lo, hi) in enumerate(wins)]
    ws_t = torch.empty(bd.bdlm_attn_fwd_tasks_workspace_bytes(tasks), dtype=torch.uint8, device="cuda")
    so = torch.empty((len(wins), L, H, d), dtype=torch.bfloat16, device="cuda")
    sl = torch.empty((len(wins), H, L), dtype=torch.float32, device="cuda")

    def step():
        for (lo, hi), po, pl in zip(wins, parts, plse):
            bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], block, part=bd.Partial.window(lo, hi), out=po, lse=pl,
                             workspace=wsf)
        bd.bdlm_lse_merge(parts, plse, out=o, lse=lse)
        bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block, dq=dq, dk=dk, dv=dv, workspace=wsb)
        bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, block, tasks, len(wins), out=so, lse=sl, workspace=ws_t)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (101, 102):
        _, y = gen(n, block, H, Hk, d, seed=seed)
        for dst, src in ((x.q, y.q), (x.k, y.k), (x.v, y.v), (x.do, y.do)):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv, so, sl)]
        step()  # the same step, eagerly
        torch.cuda.synchronize()
        ref = (o, lse, dq, dk, dv, so, sl)
        for nm, a, b in zip(("o", "lse", "dk", "dv", "slots o", "slots lse"), [got[i] for i in (0, 1, 3, 4, 5, 6)],
                            [ref[i] for i in (0, 1, 3, 4, 5, 6)]):
            assert torch.equal(a, b), f"replay {seed}: {nm} differs from the eager step"
        rel = ((got[2].float() - dq.float()).norm() / dq.float().norm()).item()
        assert rel <= 1e-3, f"replay {seed}: dq {rel:.2e}"  # fp32 reduce-adds in another order
        r = ref_full(y, w)
        check_o(host(o), r["o"], "o")
        check_grad(host(dq), r["dq"], "dq")


@pytest.mark.parametrize("n,block,H,Hk,d,groups", [(300, 32, 4, 2, 128, 3), (200, 48, 2, 1, 128, 2),
                                                   (100, 16, 2, 2, 64, 3), (150, 200, 2, 1, 128, 1)])
def test_block_groups_with_a_short_last_block(bd, n, block, H, Hk, d, groups):
    # B does not divide n: a group listing the short last block gives it B rows
    # of q, k, v, the rows past the half's end being zero padding; the forward
    # takes the list in any order, the backward ascending
    w, x = gen(n, block, H, Hk, d, seed=19 + n)
    nb = -(-n // block)
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    ws = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(2 * n, H, d, 1), dtype=torch.uint8, device="cuda")
    lists = synth.early_late_groups(nb, groups)
    assert any(nb - 1 in b for b in lists)

    def take(t, pos):  # rows at positions `pos`, zeros for padding (-1)
        p = torch.from_numpy(pos).cuda()
        out = t[p.clamp(min=0)].clone()
        out[p < 0] = 0
        return out.contiguous()

    def take64(t, pos):
        return np.where((pos >= 0)[:, None, None], t[np.maximum(pos, 0)], 0.0)

    for blocks in lists:
        for order in (blocks, blocks[::-1]):
            qpos, kpos = oracle.group_positions(n, block, order)
            part = bd.Partial.group(torch.tensor(order, dtype=torch.int32, device="cuda"))
            qg, kg, vg, dog = take(x.q, qpos), take(x.k, kpos), take(x.v, kpos), take(x.do, qpos)
            go, gl = bd.bdlm_attn_fwd(qg, kg, vg, block, L=2 * n, part=part)
            torch.cuda.synchronize()
            r = oracle.group_attention(take64(q64, qpos), take64(k64, kpos), take64(v64, kpos), n, block, order,
                                       w.scale, do=take64(do64, qpos))
            check_o(host(go), r["o"], f"group {order} o")
            check_lse(host(gl), r["lse"], f"group {order} lse")
            real = torch.from_numpy(qpos >= 0).cuda()
            assert torch.all(go[~real] == 0) and torch.all(torch.isneginf(gl[:, ~real]))
            assert (go[real].float() - o[torch.from_numpy(qpos[qpos >= 0]).cuda()].float()).abs().max() <= 2e-2
            if order != sorted(order):
                continue
            dq, dk, dv = bd.bdlm_attn_bwd(qg, kg, vg, go, gl, dog, block, L=2 * n, part=part, workspace=ws)
            assert bd.bdlm_read_error(ws) == 0
            check_grad(host(dq), r["dq"], f"group {order} dq")
            check_grad(host(dk), r["dk"], f"group {order} dk")
            check_grad(host(dv), r["dv"], f"group {order} dv")
            pad_k = torch.from_numpy(kpos < 0).cuda()
            assert torch.all(dq[~real] == 0) and torch.all(dk[pad_k] == 0) and torch.all(dv[pad_k] == 0)


def offset_moves(q, k, scale, n, block, G):
    """Moves of the forward's lazy offset after an item's first 128-key tile,
    replayed on the host for the last clean row of every head: the offset
    moves when a tile's maximum log2 score exceeds it by more than 8."""
    row, moves = n - 1, 0
    for h in range(q.shape[1]):
        s = q[row, h] @ k[:(row // block + 1) * block, h // G].T * scale / np.log(2.0)
        m = -np.inf
        for t in range(0, len(s), 128):
            mx = s[t:t + 128].max()
            if mx > m + 8:
                moves += t > 0
                m = mx
    return moves


@pytest.mark.parametrize("n,block,H,Hk,d,top", [(320, 32, 4, 2, 128, 6.0), (400, 8, 2, 1, 64, 8.0),
                                                  (512, 64, 4, 4, 128, 3.0)])
def test_growing_scores_move_the_softmax_offset(bd, n, block, H, Hk, d, top):
    """Keys whose magnitude grows along the sequence (k row t scaled by
    1 + top * t / 2n, q and k drawn with std 2) give later key tiles much
    larger row maxima, so the forward's running offset moves and O is
    rescaled in TMEM on many key tiles after an item's first, with scores
    spanning over a hundred units of log2 (3 to 7 moves on the last clean
    rows over ten seeds of each case). v is scaled back to std 0.5, so that
    o stays in the range the max-abs tolerance is stated for (bf16 rounding
    of |o| near 8 alone is up to 0.03). o, lse and the gradients against the
    float64 oracle on the same bf16 values."""
    w, x = gen(n, block, H, Hk, d, seed=n + 5, std=2.0)
    L = x.k.shape[0]
    ramp = 1.0 + top * torch.arange(L, device=x.k.device, dtype=torch.float32) / L
    x.k.copy_((x.k.float() * ramp[:, None, None]).to(x.k.dtype))
    x.v.copy_((x.v.float() * 0.25).to(x.v.dtype))
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block)
    torch.cuda.synchronize()
    r = ref_full(x, w)
    assert offset_moves(host(x.q), host(x.k), w.scale, n, block, H // Hk) > 0  # the case is what it claims
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")


@pytest.mark.parametrize("n,block,H,Hk,d,scale", [(160, 16, 4, 2, 128, 0.3), (96, 32, 2, 1, 64, 0.05)])
def test_explicit_softmax_scale(bd, n, block, H, Hk, d, scale):
    """A softmax scale other than 1/sqrt(d) reaches the forward's exponent,
    the backward's recomputed P and dS, and the dq conversion: o, lse and
    the gradients against the oracle taken with the same scale. A scale <= 0
    means 1/sqrt(d): bit-identical to the default call."""
    w, x = gen(n, block, H, Hk, d, seed=n + 11)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, block, softmax_scale=scale)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, block, softmax_scale=scale)
    torch.cuda.synchronize()
    r = oracle.bdlm_attention(host(x.q), host(x.k), host(x.v), block, scale, do=host(x.do))
    check_o(host(o), r["o"])
    check_lse(host(lse), r["lse"])
    check_grad(host(dq), r["dq"], "dq")
    check_grad(host(dk), r["dk"], "dk")
    check_grad(host(dv), r["dv"], "dv")
    o0, lse0 = bd.bdlm_attn_fwd(x.q, x.k, x.v, block)
    o1, lse1 = bd.bdlm_attn_fwd(x.q, x.k, x.v, block, softmax_scale=-1.0)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("n,block,H,Hk,d,shards", [(320, 32, 4, 2, 128, 3), (192, 16, 2, 1, 64, 4)])
def test_sharded_with_growing_scores(bd, n, block, H, Hk, d, shards):
    """Sharp scores across shards (keys growing along the sequence, as in
    test_growing_scores_move_the_softmax_offset): the windows' partial lse
    values differ by tens of log2 units row by row, so the LSE merge (of
    bf16 partials) and the forward's running merge (fp32) weigh partials
    whose weights differ by many orders of magnitude; then the sharded
    backward with the merged o and lse. All against the oracle."""
    w, x = gen(n, block, H, Hk, d, seed=7 * n + shards, std=2.0)
    L = x.k.shape[0]
    ramp = 1.0 + 6.0 * torch.arange(L, device=x.k.device, dtype=torch.float32) / L
    x.k.copy_((x.k.float() * ramp[:, None, None]).to(x.k.dtype))
    x.v.copy_((x.v.float() * 0.25).to(x.v.dtype))
    q64, k64, v64, do64 = host(x.q), host(x.k), host(x.v), host(x.do)
    full = oracle.bdlm_attention(q64, k64, v64, block, w.scale, do=do64)
    windows = synth.shard_bounds(n, shards) + [(n, 2 * n)]
    parts, lses = [], []
    o_run = torch.empty(x.q.shape, dtype=torch.float32, device="cuda")
    lse_run = torch.empty((H, 2 * n), dtype=torch.float32, device="cuda")
    for i, (lo, hi) in enumerate(windows):
        kw, vw = x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous()
        po, pl = bd.bdlm_attn_fwd(x.q, kw, vw, block, part=bd.Partial.window(lo, hi))
        parts.append(po)
        lses.append(pl)
        bd.bdlm_attn_fwd(x.q, kw, vw, block, part=bd.Partial.window(lo, hi, accumulate=i > 0), out=o_run, lse=lse_run)
    spread = torch.stack(lses)
    fin = torch.isfinite(spread)
    gap = (spread.masked_fill(~fin, -1e30).amax(0) - spread.masked_fill(~fin, 1e30).amin(0))[fin.sum(0) > 1]
    assert gap.max().item() / math.log(2.0) > 20  # partials of one row many orders of magnitude apart
    mo, ml = bd.bdlm_lse_merge(parts, lses)
    torch.cuda.synchronize()
    check_o(host(mo), full["o"], "merged o")
    check_lse(host(ml), full["lse"], "merged lse")
    check_o(host(o_run), full["o"], "running-merge o")
    check_lse(host(lse_run), full["lse"], "running-merge lse")
    dq_sum = torch.zeros(2 * n, H, d, dtype=torch.float32, device="cuda")
    dk_cat, dv_cat = torch.empty_like(x.k), torch.empty_like(x.v)
    for lo, hi in windows:
        dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k[lo:hi].contiguous(), x.v[lo:hi].contiguous(), mo, ml, x.do, block,
                                      part=bd.Partial.window(lo, hi))
        dq_sum += dq.float()
        dk_cat[lo:hi] = dk
        dv_cat[lo:hi] = dv
    torch.cuda.synchronize()
    check_grad(host(dq_sum), full["dq"], "sum of dq shares")
    check_grad(host(dk_cat), full["dk"], "dk over all shards")
    check_grad(host(dv_cat), full["dv"], "dv over all shards")
