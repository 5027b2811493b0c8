"""Pins of the float64 oracle against things other than itself: a hand-worked
example, closed forms, textbook attention in special cases, finite
differences, gradient identities, the separability and shard-merge
invariants the papers state, and a second loop-by-loop implementation."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import naive
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def case(n, block, H, Hk, d, seed=0, std=1.0):
    T = 2 * n
    q = rnd((T, H, d), seed, std)
    k = rnd((T, Hk, d), seed + 1, std)
    v = rnd((T, Hk, d), seed + 2, std)
    do = rnd((T, H, d), seed + 3)
    return q, k, v, do


# --------------------------------------------------------------------------
# mask structure
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,block", [(8, 1), (8, 2), (8, 8), (48, 16), (64, 4),
                                     (10, 4), (7, 3), (5, 8), (13, 4)])  # ragged: B does not divide n
def test_mask_population_closed_form(n, block):
    m = oracle.full_mask(n, block)
    assert int(m.sum()) == oracle.valid_pairs(n, block)
    if n % block == 0:
        assert int(m.sum()) == n * (n + block)
    rows = np.arange(2 * n)
    blk = np.where(rows < n, rows, rows - n) // block
    # every row sees (its block + 1) * B keys, capped at n (the last block may be short)
    assert np.array_equal(m.sum(axis=1), np.minimum((blk + 1) * block, n))
    # clean rows never see corrupted keys
    assert not m[:n, n:].any()
    # a corrupted key is seen only by the corrupted rows of its own block
    for j in range(n, 2 * n):
        seers = np.nonzero(m[:, j])[0]
        assert np.array_equal(seers, n + blk[j] * block + np.arange(min(block, n - blk[j] * block)))


@pytest.mark.parametrize("n,block", [(6, 1), (6, 2), (6, 3), (8, 4), (7, 3), (5, 2)])
def test_mask_matches_pairwise_rule(n, block):
    m = oracle.full_mask(n, block)
    for i in range(2 * n):
        for j in range(2 * n):
            assert m[i, j] == naive.sees(i, j, n, block), (i, j)


# --------------------------------------------------------------------------
# hand-worked golden example
# --------------------------------------------------------------------------
def test_hand_worked_example():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        g = json.load(f)
    a = np.array(g["a"])
    vv = np.array(g["v"])
    q = np.ones((4, 1, 1))
    k = np.log(a).reshape(4, 1, 1)
    v = vv.reshape(4, 1, 1)
    for c in g["cases"]:
        out = oracle.bdlm_attention(q, k, v, c["block"], 1.0)
        np.testing.assert_allclose(np.exp(out["lse"][0]), c["lse_exp"], rtol=1e-13)
        np.testing.assert_allclose(out["o"][:, 0, 0], c["o"], rtol=1e-13)


# --------------------------------------------------------------------------
# two independent oracles; block driver vs whole-mask driver
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,block", [(8, 1), (8, 2), (8, 4), (7, 3), (5, 4)])
def test_vectorised_matches_scalar_loops(n, block):
    H, Hk, d = 2, 1, 4
    q, k, v, _ = case(n, block, H, Hk, d, seed=10)
    scale = 0.7
    o_ref, lse_ref = naive.forward(q.tolist(), k.tolist(), v.tolist(), n, block, scale)
    out = oracle.bdlm_attention(q, k, v, block, scale)
    np.testing.assert_allclose(out["o"], np.array(o_ref), atol=1e-12)
    np.testing.assert_allclose(out["lse"], np.array(lse_ref), atol=1e-12)


@pytest.mark.parametrize("n,block,H,Hk", [(32, 8, 4, 2), (24, 4, 2, 2), (16, 16, 3, 1), (30, 8, 2, 1), (21, 4, 2, 2)])
def test_block_driver_matches_whole_mask(n, block, H, Hk):
    q, k, v, do = case(n, block, H, Hk, 8, seed=20)
    a = oracle.bdlm_attention(q, k, v, block, 0.35, do=do)
    b = oracle.dense_bdlm_attention(q, k, v, n, block, 0.35, do=do)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(a[key], b[key], atol=1e-12, err_msg=key)


# --------------------------------------------------------------------------
# special cases that reduce to textbook attention
# --------------------------------------------------------------------------
def _sdpa(q, k, v, scale, causal):
    # torch float64 SDPA as the textbook routine: [R,H,d] -> [1,H,R,d]
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x.transpose(1, 0, 2)))[None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal, scale=scale)
    return o[0].numpy().transpose(1, 0, 2)


def test_block_one_clean_half_is_causal_attention():
    n, H, d = 24, 2, 8
    q, k, v, _ = case(n, 1, H, H, d, seed=30)
    out = oracle.bdlm_attention(q, k, v, 1, 0.4)
    ref = _sdpa(q[:n], k[:n], v[:n], 0.4, causal=True)
    np.testing.assert_allclose(out["o"][:n], ref, atol=1e-12)
    # corrupted row of block 0 sees only itself
    np.testing.assert_allclose(out["o"][n], v[n], atol=1e-12)
    np.testing.assert_allclose(out["lse"][:, n], 0.4 * (q[n] * k[n]).sum(-1), atol=1e-12)


def test_single_block_is_bidirectional_attention_per_half():
    n, H, d = 16, 2, 8
    q, k, v, _ = case(n, n, H, H, d, seed=31)
    out = oracle.bdlm_attention(q, k, v, n, 0.3)
    np.testing.assert_allclose(out["o"][:n], _sdpa(q[:n], k[:n], v[:n], 0.3, False), atol=1e-12)
    np.testing.assert_allclose(out["o"][n:], _sdpa(q[n:], k[n:], v[n:], 0.3, False), atol=1e-12)


@pytest.mark.parametrize("n,block", [(32, 8), (30, 8)])
def test_zero_keys_closed_form(n, block):
    H, d = 2, 4
    q, _, v, _ = case(n, block, H, H, d, seed=32)
    k = np.zeros((2 * n, H, d))
    out = oracle.bdlm_attention(q, k, v, block, 0.5)
    for i in range(2 * n):
        b = (i % n) // block
        hi = min((b + 1) * block, n)  # a last block may be short
        np.testing.assert_allclose(out["lse"][:, i], math.log(hi), atol=1e-13)
        if i < n:
            vis = np.arange(0, hi)
        else:
            vis = np.concatenate([np.arange(0, b * block), n + np.arange(b * block, hi)])
        np.testing.assert_allclose(out["o"][i], v[vis].mean(axis=0), atol=1e-13)


# --------------------------------------------------------------------------
# gradients: finite differences and identities
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,block", [(8, 1), (8, 2), (8, 4), (7, 3)])
def test_finite_difference_gradients(n, block):
    H, Hk, d = 2, 1, 4
    q, k, v, do = case(n, block, H, Hk, d, seed=40)
    scale = 0.6
    g = oracle.dense_bdlm_attention(q, k, v, n, block, scale, do=do)

    def loss(q, k, v):
        return float((oracle.dense_bdlm_attention(q, k, v, n, block, scale)["o"] * do).sum())

    h = 1e-6
    for name, arr, grad in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            fd[idx] = (loss(**args_p) - loss(**args_m)) / (2 * h)
        rel = np.linalg.norm(fd - grad) / np.linalg.norm(grad)
        assert rel < 1e-6, (name, rel)


def test_gradient_identities():
    # sum_j dS_ij = 0 for every row, so the dK of all keys of a kv head sums to
    # zero; sum_j P_ij = 1, so the dV of all keys sums to the group's dO.
    n, block, H, Hk, d = 40, 8, 4, 2, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=41)
    g = oracle.bdlm_attention(q, k, v, block, 0.3, do=do)
    np.testing.assert_allclose(g["dk"].sum(axis=0), 0.0, atol=1e-11)
    G = H // Hk
    for kv in range(Hk):
        np.testing.assert_allclose(g["dv"][:, kv].sum(axis=0), do[:, kv * G:(kv + 1) * G].sum(axis=(0, 1)),
                                   atol=1e-11)


# --------------------------------------------------------------------------
# separability over target blocks (Block Parallelism abstract)
# --------------------------------------------------------------------------
def test_separability_over_blocks():
    n, block, H, Hk, d = 32, 8, 4, 2, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=50)
    scale = 0.35
    full = oracle.dense_bdlm_attention(q, k, v, n, block, scale, do=do)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(n // block):
        # clean block b alone: keys clean[0:(b+1)B], no mask
        rows = np.arange(b * block, (b + 1) * block)
        keys = np.arange(0, (b + 1) * block)
        alone = np.ones((len(rows), len(keys)), bool)
        o, lse = oracle.attend(q[rows], k[keys], v[keys], alone, scale)
        dq_b, dk_b, dv_b = oracle.attend_bwd(q[rows], k[keys], v[keys], alone, scale, o, lse, do[rows])
        np.testing.assert_allclose(o, full["o"][rows], atol=1e-12)
        np.testing.assert_allclose(lse, full["lse"][:, rows], atol=1e-12)
        np.testing.assert_allclose(dq_b, full["dq"][rows], atol=1e-12)
        dk[keys] += dk_b
        dv[keys] += dv_b
        # corrupted block b alone: keys clean[0:bB] + its own corrupted rows
        rows = n + np.arange(b * block, (b + 1) * block)
        keys = np.concatenate([np.arange(0, b * block), rows])
        alone = np.ones((len(rows), len(keys)), bool)
        o, lse = oracle.attend(q[rows], k[keys], v[keys], alone, scale)
        dq_b, dk_b, dv_b = oracle.attend_bwd(q[rows], k[keys], v[keys], alone, scale, o, lse, do[rows])
        np.testing.assert_allclose(o, full["o"][rows], atol=1e-12)
        np.testing.assert_allclose(lse, full["lse"][:, rows], atol=1e-12)
        np.testing.assert_allclose(dq_b, full["dq"][rows], atol=1e-12)
        dk[keys] += dk_b
        dv[keys] += dv_b
    np.testing.assert_allclose(dk, full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, full["dv"], atol=1e-12)


# --------------------------------------------------------------------------
# sharded clean K/V + LSE merge == unsharded (CSBP keeps the semantics)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shards", [1, 2, 3, 8])
def test_shard_then_merge_equals_unsharded(shards):
    n, block, H, Hk, d = 48, 8, 4, 2, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=60)
    scale = 0.3
    full = oracle.dense_bdlm_attention(q, k, v, n, block, scale, do=do)
    windows = synth.shard_bounds(n, shards) + [(n, 2 * n)]
    os_, lses = [], []
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for lo, hi in windows:
        p = oracle.partial_attention(q, k[lo:hi], v[lo:hi], n, block, lo, hi, scale,
                                     do=do, o_full=full["o"], lse_full=full["lse"])
        os_.append(p["o"])
        lses.append(p["lse"])
        dq += p["dq"]
        dk[lo:hi] += p["dk"]
        dv[lo:hi] += p["dv"]
    if shards > 1:
        # a late clean shard leaves early rows with no visible key
        assert np.isneginf(lses[-2]).any()
        assert np.all(os_[-2][np.isneginf(lses[-2]).T] == 0.0)
    o, lse = oracle.lse_merge(os_, lses)
    np.testing.assert_allclose(o, full["o"], atol=1e-12)
    np.testing.assert_allclose(lse, full["lse"], atol=1e-12)
    np.testing.assert_allclose(dq, full["dq"], atol=1e-12)
    np.testing.assert_allclose(dk, full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, full["dv"], atol=1e-12)


@pytest.mark.parametrize("n,block", [(48, 8), (45, 8)])
def test_row_range_by_key_window_grid(n, block):
    # Token-level tasks: any partition of the query rows by any partition of
    # the keys; per row range, merging its key windows gives the unsharded
    # attention rows and dq; dk, dv summed over every task give the unsharded
    # key gradients.
    H, Hk, d = 4, 2, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=62)
    scale = 0.3
    full = oracle.dense_bdlm_attention(q, k, v, n, block, scale, do=do)
    row_cuts = [0, 7, n - 3, n, n + 13, 2 * n]
    key_cuts = [0, 11, n - 5, n, n + 20, 2 * n]
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for qa, qb in zip(row_cuts[:-1], row_cuts[1:]):
        os_, ls_ = [], []
        dq = np.zeros((qb - qa,) + q.shape[1:])
        for ka, kb in zip(key_cuts[:-1], key_cuts[1:]):
            p = oracle.partial_attention(q[qa:qb], k[ka:kb], v[ka:kb], n, block, ka, kb, scale, do=do[qa:qb],
                                         o_full=full["o"][qa:qb], lse_full=full["lse"][:, qa:qb], q_lo=qa, q_hi=qb)
            os_.append(p["o"])
            ls_.append(p["lse"])
            dq += p["dq"]
            dk[ka:kb] += p["dk"]
            dv[ka:kb] += p["dv"]
        o, lse = oracle.lse_merge(os_, ls_)
        np.testing.assert_allclose(o, full["o"][qa:qb], atol=1e-12)
        np.testing.assert_allclose(lse, full["lse"][:, qa:qb], atol=1e-12)
        np.testing.assert_allclose(dq, full["dq"][qa:qb], atol=1e-12)
    np.testing.assert_allclose(dk, full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, full["dv"], atol=1e-12)


def test_task_list_over_packed_sequences():
    # Token-level tasks over two packed sequences of different (ragged) lengths:
    # each sequence's rows cut into row ranges and its keys into windows, task
    # (range, window w) writing slot w; per sequence, merging the slots gives
    # that sequence's attention alone, and the row ranges no task of a slot
    # covers keep their sentinel.
    H, Hk, d, block = 4, 2, 8, 4
    scale = 0.4
    ns = [13, 22]
    rows = 2 * sum(ns)
    rng = np.random.default_rng(81)
    q = rng.standard_normal((rows, H, d))
    k = rng.standard_normal((rows, Hk, d))
    v = rng.standard_normal((rows, Hk, d))
    starts = [0, 2 * ns[0]]
    tasks, n_slots = [], 3
    for s0, n in zip(starts, ns):
        row_cuts = [0, 5, n + 2, 2 * n]
        key_cuts = [0, n - 3, n + 1, 2 * n]
        for qa, qb in zip(row_cuts[:-1], row_cuts[1:]):
            for w, (ka, kb) in enumerate(zip(key_cuts[:-1], key_cuts[1:])):
                tasks.append(dict(seq_start=s0, n=n, q_lo=qa, q_hi=qb, key_lo=ka, key_hi=kb, slot=w))
    o, lse = oracle.task_attention(q, k, v, block, scale, tasks, n_slots)
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    om, lm = oracle.lse_merge(o, lse)
    for s0, n in zip(starts, ns):
        alone = oracle.dense_bdlm_attention(q[s0:s0 + 2 * n], k[s0:s0 + 2 * n], v[s0:s0 + 2 * n], n, block, scale)
        np.testing.assert_allclose(om[s0:s0 + 2 * n], alone["o"], atol=1e-12)
        np.testing.assert_allclose(lm[:, s0:s0 + 2 * n], alone["lse"], atol=1e-12)
    # the clean rows of a sequence see no corrupted key: o = 0, lse = -inf there
    n = ns[1]
    s0 = starts[1]
    t = [dict(seq_start=s0, n=n, q_lo=0, q_hi=n, key_lo=n, key_hi=2 * n, slot=1)]
    o2, l2 = oracle.task_attention(q, k, v, block, scale, t, 2)
    assert np.all(o2[1, s0:s0 + n] == 0.0) and np.all(l2[1, :, s0:s0 + n] == -np.inf)
    assert np.isnan(o2[0]).all() and np.isnan(o2[1, :s0]).all() and np.isnan(o2[1, s0 + n:]).all()


def test_task_list_backward_over_packed_sequences():
    # The backward of a task grid over two packed ragged sequences, each task
    # with the full softmax of its rows: dq summed over the tasks and dk, dv
    # summed over the slots (one slot per row range) give each sequence's
    # unsharded gradients.
    H, Hk, d, block = 4, 2, 8, 4
    scale = 0.35
    ns = [11, 18]
    rows = 2 * sum(ns)
    rng = np.random.default_rng(83)
    q = rng.standard_normal((rows, H, d))
    k = rng.standard_normal((rows, Hk, d))
    v = rng.standard_normal((rows, Hk, d))
    do = rng.standard_normal((rows, H, d))
    starts = [0, 2 * ns[0]]
    full_o = np.zeros((rows, H, d))
    full_lse = np.zeros((H, rows))
    alone = []
    for s0, n in zip(starts, ns):
        sl = slice(s0, s0 + 2 * n)
        a = oracle.dense_bdlm_attention(q[sl], k[sl], v[sl], n, block, scale, do=do[sl])
        full_o[sl], full_lse[:, sl] = a["o"], a["lse"]
        alone.append(a)
    tasks = []
    for s0, n in zip(starts, ns):
        row_cuts = [0, 6, n + 1, 2 * n]
        key_cuts = [0, n - 2, n + 3, 2 * n]
        for r, (qa, qb) in enumerate(zip(row_cuts[:-1], row_cuts[1:])):
            for ka, kb in zip(key_cuts[:-1], key_cuts[1:]):
                tasks.append(dict(seq_start=s0, n=n, q_lo=qa, q_hi=qb, key_lo=ka, key_hi=kb, slot=r))
    dq, dk, dv = oracle.task_attention_bwd(q, k, v, full_o, full_lse, do, block, scale, tasks, 3)
    assert not np.isnan(dk).any() and not np.isnan(dv).any()
    for (s0, n), a in zip(zip(starts, ns), alone):
        sl = slice(s0, s0 + 2 * n)
        np.testing.assert_allclose(dq[sl], a["dq"], atol=1e-12)
        np.testing.assert_allclose(dk[:, sl].sum(axis=0), a["dk"], atol=1e-12)
        np.testing.assert_allclose(dv[:, sl].sum(axis=0), a["dv"], atol=1e-12)


def test_merge_special_cases():
    rng = np.random.default_rng(70)
    R, H, d = 5, 2, 3
    o1 = rng.standard_normal((R, H, d))
    l1 = rng.standard_normal((H, R))
    # one partial: identity
    o, l = oracle.lse_merge([o1], [l1])
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, l1, atol=1e-15)
    # a -inf partial is dropped even if its o holds NaN
    junk = np.full((R, H, d), np.nan)
    o, l = oracle.lse_merge([o1, junk], [l1, np.full((H, R), -np.inf)])
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, l1, atol=1e-15)
    # all -inf: zero output, -inf lse
    o, l = oracle.lse_merge([junk, junk], [np.full((H, R), -np.inf)] * 2)
    assert np.all(o == 0.0) and np.all(np.isneginf(l))
    # equal lse: plain average, lse + ln 2
    o2 = rng.standard_normal((R, H, d))
    o, l = oracle.lse_merge([o1, o2], [l1, l1])
    np.testing.assert_allclose(o, (o1 + o2) / 2, atol=1e-14)
    np.testing.assert_allclose(l, l1 + math.log(2), atol=1e-14)


@pytest.mark.parametrize("shards", [2, 3, 8])
def test_running_merge_equals_one_shot_merge(shards):
    # Merging window partials one at a time into a running (o, lse), as the
    # forward's accumulate mode does, gives the one-shot merge (log-sum-exp
    # merging is associative) and so the unsharded attention; a window a row
    # cannot see (-inf partial) leaves the running row as it was.
    n, block, H, Hk, d = 48, 8, 4, 2, 8
    q, k, v, _ = case(n, block, H, Hk, d, seed=61)
    scale = 0.3
    windows = synth.shard_bounds(n, shards) + [(n, 2 * n)]
    parts = [oracle.partial_attention(q, k[lo:hi], v[lo:hi], n, block, lo, hi, scale) for lo, hi in windows]
    o, lse = parts[0]["o"], parts[0]["lse"]
    for p in parts[1:]:
        before_o, before_l = o, lse
        o, lse = oracle.lse_merge([o, p["o"]], [lse, p["lse"]])
        unseen = np.isneginf(p["lse"])
        assert np.array_equal(lse[unseen], before_l[unseen])
        assert np.array_equal(o[unseen.T], before_o[unseen.T])
    o1, lse1 = oracle.lse_merge([p["o"] for p in parts], [p["lse"] for p in parts])
    np.testing.assert_allclose(o, o1, atol=1e-12)
    np.testing.assert_allclose(lse, lse1, atol=1e-12)
    full = oracle.dense_bdlm_attention(q, k, v, n, block, scale)
    np.testing.assert_allclose(o, full["o"], atol=1e-12)
    np.testing.assert_allclose(lse, full["lse"], atol=1e-12)


# --------------------------------------------------------------------------
# early/late block groups == unsplit corrupted rows
# --------------------------------------------------------------------------
def test_block_groups_equal_unsplit():
    n, block, H, Hk, d = 64, 4, 4, 2, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=80)
    scale = 0.3
    full = oracle.bdlm_attention(q, k, v, block, scale, do=do)
    groups = synth.early_late_groups(n // block, 4)
    assert sorted(sum(groups, [])) == list(range(n // block))
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for blocks in groups:
        qpos, kpos = oracle.group_positions(n, block, blocks)
        g = oracle.group_attention(q[qpos], k[kpos], v[kpos], n, block, blocks, scale, do=do[qpos])
        np.testing.assert_allclose(g["o"], full["o"][qpos], atol=1e-12)
        np.testing.assert_allclose(g["lse"], full["lse"][:, qpos], atol=1e-12)
        np.testing.assert_allclose(g["dq"], full["dq"][qpos], atol=1e-12)
        np.add.at(dk, kpos, g["dk"])
        np.add.at(dv, kpos, g["dv"])
    # the clean rows' own contribution completes the clean keys' gradients
    clean = oracle.bdlm_attention(q, k, v, block, scale, do=do,
                                  row_blocks=[(0, b * block) for b in range(n // block)])
    np.testing.assert_allclose(dk + clean["dk"], full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv + clean["dv"], full["dv"], atol=1e-12)


def test_block_groups_with_a_short_last_block():
    # n = 62, B = 8: the last block of each half holds 6 rows. A group that
    # lists it carries 2 padding rows (and keys) in its place: they take no
    # part, and the real rows equal the unsplit rows.
    n, block, H, Hk, d = 62, 8, 2, 1, 8
    q, k, v, do = case(n, block, H, Hk, d, seed=85)
    scale = 0.3
    nb = -(-n // block)
    full = oracle.bdlm_attention(q, k, v, block, scale, do=do)
    groups = synth.early_late_groups(nb, 3)
    assert any(nb - 1 in g for g in groups)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for blocks in groups:
        qpos, kpos = oracle.group_positions(n, block, blocks)
        pad_q, pad_k = qpos < 0, kpos < 0
        assert pad_q.sum() == (2 if nb - 1 in blocks else 0)
        take = lambda t, pos: np.where((pos >= 0)[:, None, None], t[np.maximum(pos, 0)], 0.0)
        g = oracle.group_attention(take(q, qpos), take(k, kpos), take(v, kpos), n, block, blocks, scale,
                                   do=take(do, qpos))
        real = ~pad_q
        np.testing.assert_allclose(g["o"][real], full["o"][qpos[real]], atol=1e-12)
        np.testing.assert_allclose(g["lse"][:, real], full["lse"][:, qpos[real]], atol=1e-12)
        np.testing.assert_allclose(g["dq"][real], full["dq"][qpos[real]], atol=1e-12)
        assert np.all(g["o"][pad_q] == 0) and np.all(np.isneginf(g["lse"][:, pad_q])) and np.all(g["dq"][pad_q] == 0)
        assert np.all(g["dk"][pad_k] == 0) and np.all(g["dv"][pad_k] == 0)
        np.add.at(dk, kpos[~pad_k], g["dk"][~pad_k])
        np.add.at(dv, kpos[~pad_k], g["dv"][~pad_k])
    clean = oracle.bdlm_attention(q, k, v, block, scale, do=do,
                                  row_blocks=[(0, b * block) for b in range(nb)])
    np.testing.assert_allclose(dk + clean["dk"], full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv + clean["dv"], full["dv"], atol=1e-12)


# --------------------------------------------------------------------------
# packed documents: attention is confined to each document
# --------------------------------------------------------------------------
def test_packed_documents_are_independent():
    block, H, Hk, d = 4, 2, 1, 8
    lens = [16, 8, 24]
    cu = synth.cu_seqlens_of(lens)
    T = cu[-1]
    q = rnd((T, H, d), 90)
    k = rnd((T, Hk, d), 91)
    v = rnd((T, Hk, d), 92)
    do = rnd((T, H, d), 93)
    packed = oracle.bdlm_attention(q, k, v, block, 0.4, cu_seqlens=cu, do=do)
    for i, ln in enumerate(lens):
        s = slice(cu[i], cu[i + 1])
        alone = oracle.dense_bdlm_attention(q[s], k[s], v[s], ln // 2, block, 0.4, do=do[s])
        for key in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(packed[key][s], alone[key], atol=1e-12, err_msg=key)
        np.testing.assert_allclose(packed["lse"][:, s], alone["lse"], atol=1e-12)


def test_synth_workloads_are_consistent():
    w = synth.BY_NAME["packed64_b32_h32kv8_d128"]
    lens = synth.doc_lengths(w)
    assert len(lens) == 64 and all(x % 64 == 0 for x in lens)
    assert 512 <= min(lens) and max(lens) <= 32768
    g = synth.early_late_groups(16384, 16)
    assert all(len(x) == 1024 for x in g)
    assert g[0][0] == 0 and g[0][-1] == 16383
