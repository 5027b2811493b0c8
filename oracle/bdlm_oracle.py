"""Float64 CPU oracle for BDLM core attention, its backward, partial (sharded)
attention and the log-sum-exp merge.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import or call this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg
do. It shares no code with the CUDA library; both receive their inputs from
the `synth` module.

What it follows:
- Core attention is softmax(Q K^T) V with no parameters ("Efficient
  Long-context Language Model Training by Core Attention Disaggregation",
  abstract).
- The training view of a block diffusion LM: each corrupted target block sees
  the clean prefix (the correct previous blocks) and its own noised copy; the
  corrupted K/V of a block are used by that block only (rit.work blog post on
  CSBP, section on why conventional context parallelism moves extra data).
  Clean rows are autoregressive across blocks and parallel within a block
  ("Block Parallelism For Efficient Distributed Long-Context Diffusion
  Language Model Training", abstract).
- Sharding the clean sequence keeps the training semantics (same abstract), so
  attention against separate clean-K/V shards, combined by log-sum-exp
  weights, equals attention against the whole.

Readings taken where the pages are silent (each is also listed in the design
notes): clean rows see their own whole block (block-bidirectional, block-causal
across blocks); corrupted rows see clean blocks strictly before their own;
clean rows never see corrupted keys; GQA maps q head h to kv head h // (H/Hk);
lse is the natural log of sum_j exp(scale * q.k_j); a row with no visible key
has o = 0 and lse = -inf.

Every array is float64 numpy. Shapes: q/o/dq [R, H, d]; k/v/dk/dv [C, Hk, d];
lse [H, R]; mask [R, C] (rows = queries, cols = keys).
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ----------------------------------------------------------------------------
# The explicit mask (rit.work CSBP post, first section; Block Parallelism
# abstract): rows and columns are doc-local positions in [0, 2n); position p
# is clean if p < n, else corrupted; its block is (p mod n) // B.
# ----------------------------------------------------------------------------
def mask_rows(rows, n: int, block: int, cols=None) -> np.ndarray:
    """Mask rows for query positions `rows` against key positions `cols`
    (default all 2n positions) of one [clean | corrupted] sequence."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(2 * n, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
    r_clean = (rows < n)[:, None]
    c_clean = (cols < n)[None, :]
    r_blk = (np.where(rows < n, rows, rows - n) // block)[:, None]
    c_blk = (np.where(cols < n, cols, cols - n) // block)[None, :]
    clean_clean = r_clean & c_clean & (c_blk <= r_blk)
    corr_clean = (~r_clean) & c_clean & (c_blk < r_blk)
    corr_corr = (~r_clean) & (~c_clean) & (c_blk == r_blk)
    return clean_clean | corr_clean | corr_corr


def full_mask(n: int, block: int) -> np.ndarray:
    return mask_rows(np.arange(2 * n), n, block)


# ----------------------------------------------------------------------------
# Core attention on an explicit mask (Core Attention Disaggregation, abstract:
# softmax(QK^T)V), and its gradient.
# ----------------------------------------------------------------------------
def attend(q, k, v, mask, scale):
    """o = softmax(scale*q k^T restricted to mask) v, lse = ln sum exp(...).
    Rows with no visible key get o = 0 and lse = -inf."""
    R, H, d = q.shape
    Hk = k.shape[1]
    G = H // Hk
    o = np.zeros((R, H, v.shape[2]))
    lse = np.full((H, R), NEG_INF)
    for h in range(H):
        g = h // G
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        s = np.where(mask, s, NEG_INF)
        m = s.max(axis=1) if s.shape[1] else np.full(R, NEG_INF)
        live = np.isfinite(m)
        m0 = np.where(live, m, 0.0)
        e = np.exp(s - m0[:, None])
        l = e.sum(axis=1)
        with np.errstate(divide="ignore"):
            lse[h] = np.where(live, m0 + np.log(np.where(live, l, 1.0)), NEG_INF)
        p = e / np.where(live, l, 1.0)[:, None]
        o[:, h, :] = p @ v[:, g, :]
    return o, lse


def attend_bwd(q, k, v, mask, scale, o, lse, do):
    """Gradients of L = sum(do * o) for o = attend(q, k, v, mask, scale).
    Uses the row statistic D_i = sum_d do_i * o_i."""
    R, H, d = q.shape
    Hk = k.shape[1]
    G = H // Hk
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(H):
        g = h // G
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        live = np.isfinite(lse[h])
        p = np.where(mask & live[:, None], np.exp(s - np.where(live, lse[h], 0.0)[:, None]), 0.0)
        dp = do[:, h, :] @ v[:, g, :].T
        D = (do[:, h, :] * o[:, h, :]).sum(axis=1)
        ds = p * (dp - D[:, None])
        dq[:, h, :] = scale * (ds @ k[:, g, :])
        dk[:, g, :] += scale * (ds.T @ q[:, h, :])
        dv[:, g, :] += p.T @ do[:, h, :]
    return dq, dk, dv


# ----------------------------------------------------------------------------
# BDLM attention over one sequence or packed documents, one query block at a
# time: the rows of one block share one mask row, so each block gathers the
# key columns its mask row marks and attends densely on them. Memory stays
# O(B * 2n) per block however long the sequence is.
# ----------------------------------------------------------------------------
def _docs(L, cu_seqlens):
    if cu_seqlens is None:
        return [(0, L)]
    cu = [int(x) for x in cu_seqlens]
    return [(cu[i], cu[i + 1] - cu[i]) for i in range(len(cu) - 1)]


def _row_blocks(n, block):
    """(first row, rows) of every query block of one sequence, clean then
    corrupted. Blocks are cut from the start of each half, so when B does not
    divide n the last block of each half holds n mod B rows."""
    out = []
    for half in (0, n):
        for r0 in range(0, n, block):
            out.append((half + r0, min(block, n - r0)))
    return out


def _block_rows(n, block, r0):
    """Rows of the query block starting at doc-local row r0 (a block start)."""
    base = 0 if r0 < n else n
    return min(block, base + n - r0)


def bdlm_attention(q, k, v, block, scale, cu_seqlens=None, do=None,
                   row_blocks=None, want_kv_grads=True):
    """BDLM forward (and, with `do`, backward) in float64.

    q [L,H,d], k/v [L,Hk,d]; each document (or the single sequence) is
    [clean n | corrupted n]. `row_blocks`, if given, is a list of
    (doc index, doc-local first row) of the query blocks to compute; o, lse, dq
    are then valid on those rows only and dk/dv hold only their contributions.
    Inputs may be float32 arrays holding bf16 values (to save host memory at
    long lengths): every gathered block is converted to float64 before any
    arithmetic. Returns dict with o, lse and (with do) dq, dk, dv (float64).
    """
    L, H, d = q.shape
    docs = _docs(L, cu_seqlens)
    o = np.zeros(q.shape)
    lse = np.full((H, L), NEG_INF)
    grads = do is not None
    if grads:
        dq = np.zeros(q.shape)
        dk = np.zeros(k.shape)
        dv = np.zeros(v.shape)
    if row_blocks is None:
        work = []
        for di, (s0, ln) in enumerate(docs):
            for r0, _ in _row_blocks(ln // 2, block):
                work.append((di, r0))
    else:
        work = list(row_blocks)
    for di, r0 in work:
        s0, ln = docs[di]
        n = ln // 2
        rows = np.arange(r0, r0 + _block_rows(n, block, r0))
        mrow = mask_rows(rows, n, block)
        cols = np.nonzero(mrow.any(axis=0))[0]
        sub = mrow[:, cols]
        f64 = lambda x: np.asarray(x, dtype=np.float64)
        qa, ka, va = f64(q[s0 + rows]), f64(k[s0 + cols]), f64(v[s0 + cols])
        ob, lb = attend(qa, ka, va, sub, scale)
        o[s0 + rows] = ob
        lse[:, s0 + rows] = lb
        if grads:
            dqb, dkb, dvb = attend_bwd(qa, ka, va, sub, scale, ob, lb, f64(do[s0 + rows]))
            dq[s0 + rows] = dqb
            if want_kv_grads:
                np.add.at(dk, s0 + cols, dkb)
                np.add.at(dv, s0 + cols, dvb)
    out = {"o": o, "lse": lse}
    if grads:
        out.update(dq=dq, dk=dk, dv=dv)
    return out


def dense_bdlm_attention(q, k, v, n, block, scale, do=None):
    """Single-sequence BDLM attention on the whole explicit [2n, 2n] mask at
    once (small n only). Used to cross-check the block-at-a-time driver."""
    m = full_mask(n, block)
    o, lse = attend(q, k, v, m, scale)
    out = {"o": o, "lse": lse}
    if do is not None:
        dq, dk, dv = attend_bwd(q, k, v, m, scale, o, lse, do)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


# ----------------------------------------------------------------------------
# Partial attention against one key window (one clean shard, or the local
# corrupted keys), as computed per shard under context-sharded block
# parallelism (Block Parallelism abstract; rit.work post, CSBP paragraph).
# ----------------------------------------------------------------------------
def partial_attention(q, k_win, v_win, n, block, key_lo, key_hi, scale, do=None, o_full=None,
                      lse_full=None, q_lo=0, q_hi=None):
    """q holds the rows at positions [q_lo, q_hi) of one sequence (default all
    2n); k_win/v_win hold the keys at positions [key_lo, key_hi) only. Rows
    with no visible key in the window get o = 0, lse = -inf.

    With `do`, also returns the window's share of the gradients taken with the
    FULL attention's softmax (o_full, lse_full, for the same rows): dq from
    these keys only, and dk, dv of the window's keys from these rows only.
    Summed over a partition of the keys (and, for dk and dv, of the rows)
    these give the unsharded gradients.
    """
    rows = np.arange(q_lo, 2 * n if q_hi is None else q_hi)
    cols = np.arange(key_lo, key_hi)
    m = mask_rows(rows, n, block, cols)
    o, lse = attend(q, k_win, v_win, m, scale)
    out = {"o": o, "lse": lse}
    if do is not None:
        dq, dk, dv = attend_bwd(q, k_win, v_win, m, scale, o_full, lse_full, do)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


def lse_merge(os, lses):
    """Merge partials computed against disjoint key sets.

    os [P, R, H, d], lses [P, H, R]. m = max over the finite lse_p;
    w_p = exp(lse_p - m) (0 where lse_p = -inf); lse = m + ln sum w_p;
    o = sum w_p o_p / sum w_p. A row whose partials are all -inf gets o = 0,
    lse = -inf. A -inf partial is dropped by selection, so its o_p never
    enters the sum.
    """
    os = np.asarray(os, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    P, R, H, d = os.shape
    fin = np.isfinite(lses)
    m = np.where(fin, lses, NEG_INF).max(axis=0)             # [H, R]
    live = np.isfinite(m)
    m0 = np.where(live, m, 0.0)
    w = np.where(fin, np.exp(np.where(fin, lses, 0.0) - m0[None]), 0.0)  # [P, H, R]
    sw = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(live, m0 + np.log(np.where(live, sw, 1.0)), NEG_INF)
    wn = w / np.where(live, sw, 1.0)[None]                     # [P, H, R]
    o = np.zeros((R, H, d))
    for p in range(P):
        sel = fin[p].T[:, :, None]                             # [R, H, 1]
        o = o + np.where(sel, wn[p].T[:, :, None] * np.where(sel, os[p], 0.0), 0.0)
    return o, lse


# ----------------------------------------------------------------------------
# Block-group (BP) attention: the queries are the corrupted rows of a list of
# blocks, the keys are all clean rows followed by those blocks' corrupted rows
# (Block Parallelism abstract: the objective separates over target blocks;
# rit.work post: one rank owns whole target blocks and their corrupted K/V).
# ----------------------------------------------------------------------------
def group_positions(n, block, blocks):
    """Doc-local positions of a group's query rows and of its key rows. Every
    listed block takes `block` rows. When block does not divide n, the last
    block of the corrupted half is short and its rows past the half's end are
    padding, marked by position -1: they see no key and no row sees them."""
    blocks = np.asarray(blocks, dtype=np.int64)
    within = np.arange(block, dtype=np.int64)
    lens = np.minimum(block, n - blocks * block)  # rows of each listed block
    corr = n + blocks[:, None] * block + within[None, :]
    corr = np.where(within[None, :] < lens[:, None], corr, -1).reshape(-1)
    qpos = corr
    kpos = np.concatenate([np.arange(n, dtype=np.int64), corr])
    return qpos, kpos


def group_attention(q_g, k_g, v_g, n, block, blocks, scale, do=None):
    qpos, kpos = group_positions(n, block, blocks)
    m = mask_rows(np.maximum(qpos, 0), n, block, np.maximum(kpos, 0))
    m &= (qpos >= 0)[:, None] & (kpos >= 0)[None, :]  # padding rows and keys take no part
    o, lse = attend(q_g, k_g, v_g, m, scale)
    out = {"o": o, "lse": lse}
    if do is not None:
        dq, dk, dv = attend_bwd(q_g, k_g, v_g, m, scale, o, lse, do)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


# ----------------------------------------------------------------------------
# Token-level task lists ("Efficient Long-context Language Model Training by
# Core Attention Disaggregation", abstract: core attention is stateless and
# composes over fused batches of token-level shards of arbitrary lengths).
# A task is one query row range of one sequence against one key window of the
# same sequence, under that sequence's BDLM mask; its result is a partial (o,
# lse) for those rows, which a log-sum-exp merge combines with the partials of
# the same rows against other keys.
# ----------------------------------------------------------------------------
def task_attention(q, k, v, block, scale, tasks, n_slots, o=None, lse=None):
    """Run a list of tasks over packed sequences.

    q [L, H, d], k/v [L, Hk, d] hold every row. A task is a dict with
    seq_start, n (its sequence is rows [seq_start, seq_start + 2n), clean then
    corrupted), q_lo, q_hi, key_lo, key_hi (positions within the sequence) and
    slot. Task t writes the partial of its rows against its keys into
    o[slot, seq_start + q_lo : seq_start + q_hi] and the matching lse columns;
    rows no task of a slot covers keep their value in the given o / lse
    (default: NaN). Returns o [S, L, H, d], lse [S, H, L].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, H, d = q.shape
    o = np.full((n_slots, L, H, d), np.nan) if o is None else np.array(o, dtype=np.float64)
    lse = np.full((n_slots, H, L), np.nan) if lse is None else np.array(lse, dtype=np.float64)
    for t in tasks:
        s0, n = t["seq_start"], t["n"]
        qa, qb = s0 + t["q_lo"], s0 + t["q_hi"]
        ka, kb = s0 + t["key_lo"], s0 + t["key_hi"]
        r = partial_attention(q[qa:qb], k[ka:kb], v[ka:kb], n, block, t["key_lo"], t["key_hi"], scale,
                              q_lo=t["q_lo"], q_hi=t["q_hi"])
        o[t["slot"], qa:qb] = r["o"]
        lse[t["slot"], :, qa:qb] = r["lse"]
    return o, lse


def task_attention_bwd(q, k, v, o_full, lse_full, do, block, scale, tasks, n_slots):
    """Backward of a task list, each task taken with the FULL softmax of its
    rows (o_full [L, H, d], lse_full [H, L]: the merge over every key a row
    sees), as in the sharded backward.

    Returns dq [L, H, d], the sum of every task's dq share (0 on rows no task
    covers), and dk, dv [S, L, Hk, d]: task t writes the gradients of its
    window's keys from its rows into slot t (rows of k no task of a slot
    covers stay NaN). Summed over a partition of every sequence's rows x keys
    (with the tasks of one row range in one slot), dq, and dk, dv summed over
    the slots, are the unsharded gradients.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    L, H, d = q.shape
    Hk = k.shape[1]
    dq = np.zeros((L, H, d))
    dk = np.full((n_slots, L, Hk, d), np.nan)
    dv = np.full((n_slots, L, Hk, d), np.nan)
    for t in tasks:
        s0, n = t["seq_start"], t["n"]
        qa, qb = s0 + t["q_lo"], s0 + t["q_hi"]
        ka, kb = s0 + t["key_lo"], s0 + t["key_hi"]
        r = partial_attention(q[qa:qb], k[ka:kb], v[ka:kb], n, block, t["key_lo"], t["key_hi"], scale,
                              do=do[qa:qb], o_full=o_full[qa:qb], lse_full=lse_full[:, qa:qb],
                              q_lo=t["q_lo"], q_hi=t["q_hi"])
        dq[qa:qb] += r["dq"]
        dk[t["slot"], ka:kb] = r["dk"]
        dv[t["slot"], ka:kb] = r["dv"]
    return dq, dk, dv


def valid_pairs(n, block):
    """Closed form of the mask's population per head for one sequence.
    With n = nb B + r: the clean rows of a full block b see (b+1)B keys, the
    r rows of a last partial block see all n clean keys; the corrupted rows of
    a full block b see bB clean keys plus their own B corrupted keys, those of
    the partial block nb B + r = n. Each half contributes
    B^2 nb (nb + 1) / 2 + r n; when B divides n this is n (n + B) for both."""
    nb, r = divmod(n, block)
    return block * block * nb * (nb + 1) + 2 * r * n
