"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times. The float64 oracle checks, on every kv group of each
workload:
  - sampled query blocks one by one (o, lse and dq are row-local), spread
    from the first to the last block of both halves;
  - complete dk, dv of late clean key blocks and of corrupted key blocks
    (every query block that sees them is recomputed);
  - for early clean key blocks, whose complete gradient needs every row's
    full softmax (the whole forward of a kv group), the contribution of
    sampled query blocks, through the row-restricted key-window backward:
    the same kernel, asked for one query block against one key block;
and identities that hold at any size: sum_j dK_j = 0 and
sum_j dV_j = sum_i dO_i per kv head. The 256K block groups are checked
against the oracle directly (each group's earliest and latest blocks), not
only against the unsplit call."""
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


def group_slices(x, w, g):
    G = w.heads // w.kv_heads
    return x.q[:, g * G:(g + 1) * G], x.k[:, g:g + 1], x.v[:, g:g + 1], x.do[:, g * G:(g + 1) * G]


def f32(t):
    return t.float().cpu().numpy()


def host_group(x, w, g):
    """q, k, v, dO of kv group g as float32 host arrays holding the bf16 values."""
    return tuple(f32(t) for t in group_slices(x, w, g))


def sampled_rows_check(x, w, o, lse, dq, kv_groups, blocks, cu=None, hg=None):
    """o, lse, dq of the given query blocks (doc, first row) against the oracle."""
    G = w.heads // w.kv_heads
    for g in kv_groups:
        q, k, v, do = hg if hg is not None else host_group(x, w, g)
        r = oracle.bdlm_attention(q, k, v, w.block, w.scale, cu_seqlens=cu, do=do, row_blocks=blocks,
                                  want_kv_grads=False)
        starts = [0] if cu is None else cu
        rows = np.concatenate([starts[d] + np.arange(r0, r0 + w.block) for d, r0 in blocks])
        hs = slice(g * G, (g + 1) * G)
        check_o(host(o[rows][:, hs]), r["o"][rows], f"o (kv group {g})")
        check_lse(host(lse[hs][:, rows]), r["lse"][:, rows], f"lse (kv group {g})")
        check_grad(host(dq[rows][:, hs]), r["dq"][rows], f"dq (kv group {g})")
    return r


def sampled_keys_check(x, w, dk, dv, g, n, key_blocks, hg=None):
    """Complete dk, dv of the clean key block b_c (seen by clean blocks >= b_c
    and corrupted blocks > b_c) and of corrupted key blocks (seen by their own
    block), for kv group g."""
    B = w.block
    nb = n // B
    q, k, v, do = hg if hg is not None else host_group(x, w, g)
    for kind, b in key_blocks:
        if kind == "clean":
            seers = [(0, bb * B) for bb in range(b, nb)] + [(0, n + bb * B) for bb in range(b + 1, nb)]
            keys = np.arange(b * B, (b + 1) * B)
        else:
            seers = [(0, n + b * B)]
            keys = n + np.arange(b * B, (b + 1) * B)
        r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=seers)
        check_grad(host(dk[keys][:, g:g + 1]), r["dk"][keys], f"dk {kind} block {b}")
        check_grad(host(dv[keys][:, g:g + 1]), r["dv"][keys], f"dv {kind} block {b}")


def workspaces(bd, w, L, n_docs=1):
    f = torch.empty(bd.bdlm_attn_fwd_workspace_bytes(L, w.heads, w.head_dim, n_docs), dtype=torch.uint8, device="cuda")
    b = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(L, w.heads, w.head_dim, n_docs), dtype=torch.uint8, device="cuda")
    return f, b


def identities_check(x, w, dk, dv):
    G = w.heads // w.kv_heads
    dk64 = dk.double()
    s = dk64.sum(0)                                   # [Hk, d]
    scale = dk64.abs().sum(0)
    assert (s.abs() <= 1e-2 * scale + 1e-3).all(), "sum of dK over keys is not ~0"
    dv_sum = dv.double().sum(0)
    do_sum = x.do.double().view(x.do.shape[0], w.kv_heads, G, -1).sum((0, 2))
    rel = (dv_sum - do_sum).norm() / do_sum.norm()
    assert rel <= 1e-2, f"sum of dV differs from sum of dO: {rel:.3e}"


def spread_blocks(n, B, shard_rows=0):
    """16 query blocks, 8 per half: the first two, the two around the first
    clean-shard boundary (if any), two in the middle and the last two. The
    pairs straddle a 128-row forward tile boundary or sit inside one tile."""
    nb = n // B
    sh = shard_rows // B if shard_rows else nb // 4
    clean = sorted({0, 1, sh - 1, sh, nb // 2 - 1, nb // 2, nb - 2, nb - 1})
    corr = sorted({0, 1, sh - 1, sh, nb // 2, nb // 2 + 1, nb - 2, nb - 1})
    return [(0, b * B) for b in clean] + [(0, n + b * B) for b in corr]


def early_key_check(bd, x, w, o, lse, g, n, key_block, seer_blocks, ref, hg=None, ws=None):
    """Contribution of each listed query block to dk, dv of one early clean key
    block, for kv group g: the GPU's key-window backward restricted to that
    query block's rows (o, lse: the merged full forward), against the
    oracle's partial backward of the same rows and keys, taken with the
    oracle's own full-row o and lse (`ref`, an oracle result that covers
    the listed blocks)."""
    B = w.block
    lo, hi = key_block * B, (key_block + 1) * B
    q, k, v, do = hg if hg is not None else host_group(x, w, g)
    for _, r0 in seer_blocks:
        rows = slice(r0, r0 + B)
        part = oracle.partial_attention(q[rows], k[lo:hi], v[lo:hi], n, B, lo, hi, w.scale, do=do[rows],
                                        o_full=ref["o"][rows], lse_full=ref["lse"][:, rows], q_lo=r0, q_hi=r0 + B)
        _, gk, gv = bd.bdlm_attn_bwd(x.q[rows], x.k[lo:hi], x.v[lo:hi], o[rows], lse[:, rows].contiguous(),
                                     x.do[rows], B, L=2 * n, part=bd.Partial.window(lo, hi, q_lo=r0, q_hi=r0 + B),
                                     workspace=ws)
        assert ws is None or bd.bdlm_read_error(ws) == 0
        what = f"kv group {g}, key block {key_block} from rows {r0}"
        check_grad(host(gk[:, g:g + 1]), part["dk"], "dk, " + what)
        check_grad(host(gv[:, g:g + 1]), part["dv"], "dv, " + what)


def test_long128k_sharded_forward_merge_backward(bd):
    w = synth.BY_NAME["long128k_n131072_b64_h32kv8_d128"]
    x = synth.make_inputs(w, device="cuda")
    n, B = w.n, w.block
    windows = synth.shard_bounds(n, w.shards) + [(n, 2 * n)]
    wsf, wsb = workspaces(bd, w, 2 * n)
    parts, lses = [], []
    for lo, hi in windows:
        po, pl = bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], B, part=bd.Partial.window(lo, hi), workspace=wsf)
        assert bd.bdlm_read_error(wsf) == 0
        parts.append(po)
        lses.append(pl)
    o, lse = bd.bdlm_lse_merge(parts, lses)
    del parts
    uo, ul = bd.bdlm_attn_fwd(x.q, x.k, x.v, B, workspace=wsf)
    assert bd.bdlm_read_error(wsf) == 0
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, B, workspace=wsb)
    assert bd.bdlm_read_error(wsb) == 0
    # sharded + merged == unsharded (both on the GPU)
    assert (o.float() - uo.float()).abs().max().item() <= 2e-2
    assert ((lse - ul).abs() / ul.abs().clamp(min=1.0)).max().item() <= 1e-3
    del uo, ul
    # the same windows merged into a running fp32 (o, lse) by the forward's
    # epilogue == the merge kernel's result
    ro = torch.empty(x.q.shape, dtype=torch.float32, device="cuda")
    rl = torch.empty_like(lse)
    for i, (lo, hi) in enumerate(windows):
        bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], B, part=bd.Partial.window(lo, hi, accumulate=i > 0), out=ro,
                         lse=rl, workspace=wsf)
    assert bd.bdlm_read_error(wsf) == 0
    assert (ro - o.float()).abs().max().item() <= 2e-2
    assert ((rl - lse).abs() / lse.abs().clamp(min=1.0)).max().item() <= 1e-3
    del ro, rl
    nb = n // B
    # every kv group: 16 query blocks row by row; complete dk, dv of two late
    # clean and two corrupted key blocks; two early clean key blocks through
    # the contributions of query blocks from both halves
    blocks = spread_blocks(n, B, shard_rows=n // w.shards)
    for g in range(w.kv_heads):
        hg = host_group(x, w, g)
        ref = sampled_rows_check(x, w, o, lse, dq, kv_groups=[g], blocks=blocks, hg=hg)
        sampled_keys_check(x, w, dk, dv, g=g, n=n, key_blocks=[("clean", nb - 1), ("clean", nb - 2),
                                                               ("corrupted", 0), ("corrupted", nb // 2 + 1)], hg=hg)
        early_key_check(bd, x, w, o, lse, g, n, 0, [(0, 0), (0, (nb // 2) * B), (0, (nb - 1) * B), (0, n + B),
                                                    (0, n + (nb - 1) * B)], ref, hg=hg, ws=wsb)
        early_key_check(bd, x, w, o, lse, g, n, nb // 2, [(0, (nb // 2) * B), (0, n + (nb // 2 + 1) * B)], ref,
                        hg=hg, ws=wsb)
        del hg, ref
    identities_check(x, w, dk, dv)
    # sharded backward: per-shard calls with the merged o and lse; the dq
    # shares sum to the unsharded dq and the shards' dk, dv tile it
    dq_sum = torch.zeros(dq.shape, dtype=torch.float32, device="cuda")
    for lo, hi in windows:
        sq, sk, sv = bd.bdlm_attn_bwd(x.q, x.k[lo:hi], x.v[lo:hi], o, lse, x.do, B,
                                      part=bd.Partial.window(lo, hi), workspace=wsb)
        assert bd.bdlm_read_error(wsb) == 0
        dq_sum += sq.float()
        del sq
        for got, ref, nm in ((sk, dk[lo:hi], "dk"), (sv, dv[lo:hi], "dv")):
            rel = ((got.float() - ref.float()).norm() / ref.float().norm()).item()
            assert rel <= 1e-2, f"{nm} of shard [{lo},{hi}): {rel:.3e}"
    rel = ((dq_sum - dq.float()).norm() / dq.float().norm()).item()
    assert rel <= 1e-2, f"sum of dq shares: {rel:.3e}"


def test_long128k_task_lists(bd):
    # the CSBP windows of the 128K workload as one forward task list and one
    # backward task list, against the window calls and the full backward
    w = synth.BY_NAME["long128k_n131072_b64_h32kv8_d128"]
    x = synth.make_inputs(w, device="cuda")
    n, B = w.n, w.block
    windows = synth.shard_bounds(n, w.shards) + [(n, 2 * n)]
    wsf, wsb = workspaces(bd, w, 2 * n)
    tasks = [bd.Task(0, n, 0, 2 * n, lo, hi, i) for i, (lo, hi) in enumerate(windows)]
    so, sl = bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, B, tasks, len(tasks))
    torch.cuda.synchronize()
    for i, (lo, hi) in enumerate(windows):  # same tiles, same arithmetic: the same bits
        po, pl = bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], B, part=bd.Partial.window(lo, hi), workspace=wsf)
        assert bd.bdlm_read_error(wsf) == 0
        assert torch.equal(so[i], po) and torch.equal(sl[i], pl), f"window {i}"
        del po, pl
    o, lse = bd.bdlm_lse_merge([so[i] for i in range(len(tasks))], [sl[i] for i in range(len(tasks))])
    del so, sl
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, B, workspace=wsb)
    assert bd.bdlm_read_error(wsb) == 0
    bwd_tasks = [bd.Task(0, n, 0, 2 * n, lo, hi, 0) for lo, hi in windows]
    tq, tk, tv = bd.bdlm_attn_bwd_tasks(x.q, x.k, x.v, o, lse, x.do, B, bwd_tasks, 1)
    torch.cuda.synchronize()
    for got, ref, nm in ((tq, dq, "dq"), (tk[0], dk, "dk"), (tv[0], dv, "dv")):
        rel = ((got.float() - ref.float()).norm() / ref.float().norm()).item()
        assert rel <= 1e-2, f"{nm} of the backward task list: {rel:.3e}"
    # and against the oracle on sampled blocks
    nb = n // B
    blocks = [(0, (nb - 1) * B), (0, n + (nb // 2) * B)]
    sampled_rows_check(x, w, o, lse, tq, kv_groups=[5], blocks=blocks)
    sampled_keys_check(x, w, tk[0], tv[0], g=5, n=n, key_blocks=[("clean", nb - 3), ("corrupted", nb - 1)])


def test_vlong256k_block_groups_and_backward(bd):
    w = synth.BY_NAME["vlong256k_n262144_b16_h16kv4_d128"]
    x = synth.make_inputs(w, device="cuda")
    n, B = w.n, w.block
    nb = n // B
    wsf, wsb = workspaces(bd, w, 2 * n)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, B, workspace=wsf)
    assert bd.bdlm_read_error(wsf) == 0
    groups = synth.early_late_groups(nb, w.groups)
    G = w.heads // w.kv_heads
    # the oracle's o, lse, dq of each group's earliest and latest block (the
    # early/late pair that opens and closes its list), on kv group gi mod Hk
    ref_rows = {}
    for g in range(w.kv_heads):
        mine = [gi for gi in range(len(groups)) if gi % w.kv_heads == g]
        if not mine:
            continue
        q, k, v, do = host_group(x, w, g)
        for gi in mine:
            ends = (groups[gi][0], groups[gi][-1])
            r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=[(0, n + b * B) for b in ends],
                                      want_kv_grads=False)
            for b in ends:
                rows = slice(n + b * B, n + (b + 1) * B)
                ref_rows[(gi, b)] = (r["o"][rows], r["lse"][:, rows], r["dq"][rows])
        del q, k, v, do

    def group_vs_oracle(gi, blocks, t, what):
        """Rows of the group's earliest and latest block in a group call's
        output t ([list rows, H, d], or [H, list rows] for lse) against the oracle."""
        g = gi % w.kv_heads
        hs = slice(g * G, (g + 1) * G)
        for b in (blocks[0], blocks[-1]):
            li = blocks.index(b)
            lr = slice(li * B, (li + 1) * B)
            ro, rl, rq = ref_rows[(gi, b)]
            tag = f"group {gi} block {b} {what}"
            if what == "o":
                check_o(host(t[lr][:, hs]), ro, tag)
            elif what == "lse":
                check_lse(host(t[hs][:, lr]), rl, tag)
            else:
                check_grad(host(t[lr][:, hs]), rq, tag)

    worst_o, worst_l = 0.0, 0.0
    clean_pos = torch.arange(n, device="cuda")
    for gi, blocks in enumerate(groups):
        bl = torch.tensor(blocks, dtype=torch.int32, device="cuda")
        corr = (n + bl.long()[:, None] * B + torch.arange(B, device="cuda")[None]).reshape(-1)
        kpos = torch.cat([clean_pos, corr])
        go, gl = bd.bdlm_attn_fwd(x.q[corr].contiguous(), x.k[kpos].contiguous(), x.v[kpos].contiguous(), B,
                                  L=2 * n, part=bd.Partial.group(bl), workspace=wsf)
        assert bd.bdlm_read_error(wsf) == 0
        worst_o = max(worst_o, (go.float() - o[corr].float()).abs().max().item())
        worst_l = max(worst_l, ((gl - lse[:, corr]).abs() / lse[:, corr].abs().clamp(min=1.0)).max().item())
        group_vs_oracle(gi, blocks, go, "o")
        group_vs_oracle(gi, blocks, gl, "lse")
    assert worst_o <= 2e-2 and worst_l <= 1e-3, (worst_o, worst_l)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, B, workspace=wsb)
    assert bd.bdlm_read_error(wsb) == 0
    # every kv group: 16 query blocks of the unsplit call row by row, complete
    # dk, dv of late clean and of corrupted key blocks
    blocks = spread_blocks(n, B)
    for g in range(w.kv_heads):
        hg = host_group(x, w, g)
        sampled_rows_check(x, w, o, lse, dq, kv_groups=[g], blocks=blocks, hg=hg)
        sampled_keys_check(x, w, dk, dv, g=g, n=n, key_blocks=[("clean", nb - 1), ("clean", nb - 2),
                                                               ("corrupted", 5), ("corrupted", nb // 2)], hg=hg)
        del hg
    identities_check(x, w, dk, dv)
    # block-group backward of every group: dq of the group's rows and dk, dv
    # of its corrupted keys equal the unsplit backward's, and its earliest and
    # latest blocks' dq equal the oracle's; for group 0, the group's share of
    # dk, dv of a late clean key block against the oracle
    for gi, blocks in enumerate(groups):
        bl = torch.tensor(blocks, dtype=torch.int32, device="cuda")
        corr = (n + bl.long()[:, None] * B + torch.arange(B, device="cuda")[None]).reshape(-1)
        kpos = torch.cat([clean_pos, corr])
        part = bd.Partial.group(bl)
        qg, kg, vg, dog = x.q[corr].contiguous(), x.k[kpos].contiguous(), x.v[kpos].contiguous(), x.do[corr].contiguous()
        go, gl = bd.bdlm_attn_fwd(qg, kg, vg, B, L=2 * n, part=part, workspace=wsf)
        gq, gk, gv = bd.bdlm_attn_bwd(qg, kg, vg, go, gl, dog, B, L=2 * n, part=part, workspace=wsb)
        assert bd.bdlm_read_error(wsb) == 0
        for got, ref, nm in ((gq, dq[corr], "dq"), (gk[n:], dk[corr], "dk"), (gv[n:], dv[corr], "dv")):
            rel = ((got.float() - ref.float()).norm() / ref.float().norm()).item()
            assert rel <= 1e-2, f"group {gi} {nm}: {rel:.3e}"
        group_vs_oracle(gi, blocks, gq, "dq")
        if gi == 0:
            b = nb - 64  # seen by the group's blocks after it (a few late ones)
            seers = [(0, n + bb * B) for bb in blocks if bb > b]
            keys = np.arange(b * B, (b + 1) * B)
            for g in (0, w.kv_heads - 1):
                q, k, v, do = (f32(t) for t in group_slices(x, w, g))
                r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=seers)
                check_grad(host(gk[keys][:, g:g + 1]), r["dk"][keys], f"group 0 dk clean block {b}")
                check_grad(host(gv[keys][:, g:g + 1]), r["dv"][keys], f"group 0 dv clean block {b}")
        del go, gl, gq, gk, gv, qg, kg, vg, dog


def test_packed_documents_full_size(bd):
    w = synth.BY_NAME["packed64_b32_h32kv8_d128"]
    x = synth.make_inputs(w, device="cuda")
    cu = x.cu_seqlens
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    B = w.block
    wsf, wsb = workspaces(bd, w, cu[-1], len(cu) - 1)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, B, cu_seqlens=cu_d, workspace=wsf)
    assert bd.bdlm_read_error(wsf) == 0
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, B, cu_seqlens=cu_d, workspace=wsb)
    assert bd.bdlm_read_error(wsb) == 0
    lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    # two short documents in full (all gradients, one kv group)
    short = sorted(range(len(lens)), key=lambda i: lens[i])[:2]
    G = w.heads // w.kv_heads
    for d in short:
        s = slice(cu[d], cu[d + 1])
        q, k, v, do = (f32(t[s]) for t in group_slices(x, w, 2))
        r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do)
        check_o(host(o[s][:, 2 * G:3 * G]), r["o"])
        check_lse(host(lse[2 * G:3 * G, s]), r["lse"])
        check_grad(host(dq[s][:, 2 * G:3 * G]), r["dq"], "dq")
        check_grad(host(dk[s][:, 2:3]), r["dk"], "dk")
        check_grad(host(dv[s][:, 2:3]), r["dv"], "dv")
    # every kv group: the median-length document in full, and sampled blocks
    # (first, middle and last of both halves) of the longest and the median one
    order = sorted(range(len(lens)), key=lambda i: lens[i])
    big, med = order[-1], order[len(order) // 2]
    blocks = []
    for d in (big, med):
        nd = lens[d] // 2
        nbd = nd // B
        blocks += [(d, 0), (d, B), (d, (nbd // 2) * B), (d, nd - B), (d, nd), (d, nd + (nbd // 2) * B),
                   (d, 2 * nd - 2 * B), (d, 2 * nd - B)]
    sm = slice(cu[med], cu[med + 1])
    for g in range(w.kv_heads):
        sampled_rows_check(x, w, o, lse, dq, kv_groups=[g], blocks=blocks, cu=cu)
        q, k, v, do = (f32(t[sm]) for t in group_slices(x, w, g))
        r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do)
        hs = slice(g * G, (g + 1) * G)
        tag = f"median document, kv group {g}"
        check_o(host(o[sm][:, hs]), r["o"], "o, " + tag)
        check_lse(host(lse[hs, sm]), r["lse"], "lse, " + tag)
        check_grad(host(dq[sm][:, hs]), r["dq"], "dq, " + tag)
        check_grad(host(dk[sm][:, g:g + 1]), r["dk"], "dk, " + tag)
        check_grad(host(dv[sm][:, g:g + 1]), r["dv"], "dv, " + tag)
    identities_check(x, w, dk, dv)


def test_packed_documents_as_task_lists(bd):
    # the 64 packed documents as token-level tasks (each document: its rows
    # against its clean keys into slot 0 and against its corrupted keys into
    # slot 1), forward and backward in one launch each, against the varlen calls
    w = synth.BY_NAME["packed64_b32_h32kv8_d128"]
    x = synth.make_inputs(w, device="cuda")
    cu = x.cu_seqlens
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    B, L = w.block, cu[-1]
    wsf, wsb = workspaces(bd, w, L, len(cu) - 1)
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, B, cu_seqlens=cu_d, workspace=wsf)
    dq, dk, dv = bd.bdlm_attn_bwd(x.q, x.k, x.v, o, lse, x.do, B, cu_seqlens=cu_d, workspace=wsb)
    assert bd.bdlm_read_error(wsb) == 0
    tasks = []
    for i in range(len(cu) - 1):
        s0, n = int(cu[i]), int(cu[i + 1] - cu[i]) // 2
        tasks += [bd.Task(s0, n, 0, 2 * n, 0, n, 0), bd.Task(s0, n, 0, 2 * n, n, 2 * n, 1)]
    so, sl = bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, B, tasks, 2)
    mo, ml = bd.bdlm_lse_merge([so[0], so[1]], [sl[0], sl[1]])
    torch.cuda.synchronize()
    assert (mo.float() - o.float()).abs().max().item() <= 2e-2
    assert ((ml - lse).abs() / lse.abs().clamp(min=1.0)).max().item() <= 1e-3
    del so, sl
    # backward: each document's two windows have disjoint keys, so one slot holds them all
    bt = [bd.Task(t.seq_start, t.n, t.q_lo, t.q_hi, t.key_lo, t.key_hi, 0) for t in tasks]
    tq, tk, tv = bd.bdlm_attn_bwd_tasks(x.q, x.k, x.v, o, lse, x.do, B, bt, 1)
    torch.cuda.synchronize()
    for got, ref, nm in ((tq, dq, "dq"), (tk[0], dk, "dk"), (tv[0], dv, "dv")):
        rel = ((got.float() - ref.float()).norm() / ref.float().norm()).item()
        assert rel <= 1e-2, f"{nm} of the packed task list: {rel:.3e}"
    identities_check(x, w, tk[0], tv[0])
