"""Context-sharded block parallelism: the plan, and the exchange of clean K/V
and of their gradients between ranks.

- The plan (CPU): every row and every key belongs to exactly one rank, the
  ranks together compute every valid pair exactly once (n(n + B) per head),
  and early/late pairing keeps the corrupted-block work balanced.
- The exchange (CPU, gloo, 2 to 4 ranks; with 4 ranks over 2 blocks, two
  ranks own no corrupted block): each rank runs its calls through
  the float64 oracle; after the all-gather and the reduce-scatter, every
  rank's o, lse, dq of its rows and dk, dv of its keys equal the unsharded
  oracle's.
- The exchange itself (CPU, gloo, 3 ranks): bf16 shards gathered bit for
  bit, gradient shares summed.
- The CUDA library (GPU): all ranks emulated in one process, each rank's
  calls on the GPU; and two ranks as two processes sharing the GPU, with
  gloo staging the exchange through host memory. Every rank's results
  against the unsharded float64 oracle: in full on small sequences, on
  sampled blocks and key blocks at 128K.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
import synth
from block_diffusion_lm_bdlm_gb300 import csbp


class OracleOps:
    """The four calls of a rank in float64 on the CPU (test infrastructure)."""

    def __init__(self, scale):
        self.scale = scale

    @staticmethod
    def _np(t):
        return t.detach().cpu().double().numpy()

    @staticmethod
    def _t(a, like):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dtype=torch.float64, device=like.device)

    def fwd_clean(self, q, k, v, n, block, lo, hi):
        r = oracle.partial_attention(self._np(q), self._np(k), self._np(v), n, block, 0, n, self.scale, q_lo=lo,
                                     q_hi=hi)
        return self._t(r["o"], q), self._t(r["lse"], q)

    def fwd_group(self, q, k, v, n, block, blocks):
        r = oracle.group_attention(self._np(q), self._np(k), self._np(v), n, block, blocks.tolist(), self.scale)
        return self._t(r["o"], q), self._t(r["lse"], q)

    def bwd_clean(self, q, k, v, o, lse, do, n, block, lo, hi):
        r = oracle.partial_attention(self._np(q), self._np(k), self._np(v), n, block, 0, n, self.scale,
                                     do=self._np(do), o_full=self._np(o), lse_full=self._np(lse), q_lo=lo, q_hi=hi)
        return self._t(r["dq"], q), self._t(r["dk"], q), self._t(r["dv"], q)

    def bwd_group(self, q, k, v, o, lse, do, n, block, blocks):
        r = oracle.group_attention(self._np(q), self._np(k), self._np(v), n, block, blocks.tolist(), self.scale,
                                   do=self._np(do))
        return self._t(r["dq"], q), self._t(r["dk"], q), self._t(r["dv"], q)


# ----------------------------------------------------------------------------
# the plan
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("n,block,ranks", [(64, 8, 2), (96, 8, 3), (100, 8, 4), (128, 16, 8), (131072, 64, 8),
                                           (30, 7, 3)])
def test_plan_covers_every_row_key_and_pair_once(n, block, ranks):
    plan = csbp.CSBPPlan.build(n, block, ranks)
    nb = (n + block - 1) // block
    clean = np.zeros(n, dtype=int)
    blocks = np.zeros(nb, dtype=int)
    for r in range(ranks):
        p = plan.rank(r)
        assert p.clean_hi - p.clean_lo == n // ranks
        clean[p.clean_lo:p.clean_hi] += 1
        assert list(p.blocks) == sorted(p.blocks)
        for b in p.blocks:
            blocks[b] += 1
    assert (clean == 1).all() and (blocks == 1).all()
    # the ranks' valid pairs add up to the mask's population
    assert sum(plan.valid_pairs(r) for r in range(ranks)) == oracle.valid_pairs(n, block)
    if n <= 128:  # and each rank's count is the explicit mask's, row by row
        m = oracle.full_mask(n, block)
        for r in range(ranks):
            p = plan.rank(r)
            rows = list(range(p.clean_lo, p.clean_hi)) + [x for x in plan.corrupted_rows(r) if x < 2 * n]
            assert plan.valid_pairs(r) == int(m[rows].sum())


def test_early_late_pairing_balances_the_corrupted_blocks():
    n, B, R = 131072, 64, 8
    plan = csbp.CSBPPlan.build(n, B, R)
    corr = []
    for r in range(R):
        corr.append(sum(B * (b * B + B) for b in plan.rank(r).blocks))
    assert max(corr) / min(corr) < 1.001
    # pairing is what balances: the same number of blocks dealt in order
    # (rank r takes blocks r, r + R, ...) is far less even
    naive = [sum(B * (b * B + B) for b in range(r, n // B, R)) for r in range(R)]
    assert max(naive) / min(naive) > max(corr) / min(corr)


def test_plan_rejects_unequal_shards():
    with pytest.raises(ValueError):
        csbp.CSBPPlan.build(100, 8, 3)


# ----------------------------------------------------------------------------
# the exchange, gloo ranks on CPU
# ----------------------------------------------------------------------------
def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(n, block, H, Hk, d, seed):
    w = synth.Workload("csbp", n=n, block=block, heads=H, kv_heads=Hk, head_dim=d, seed=seed, qkv_std=0.5)
    x = synth.make_inputs(w, device="cpu", dtype=torch.float64)
    return w, x


def _check_rank(plan, r, x, w, f, g, ref, atol):
    p = plan.rank(r)
    n = plan.n
    rows = np.array(plan.corrupted_rows(r), dtype=np.int64)
    real = rows < 2 * n
    c = slice(p.clean_lo, p.clean_hi)

    def close(got, want, what):
        got = got.detach().cpu().double().numpy()
        assert np.allclose(got, want, atol=atol, rtol=atol), f"rank {r}: {what}"

    close(f.o_clean, ref["o"][c], "o of the clean rows")
    close(f.lse_clean, ref["lse"][:, c], "lse of the clean rows")
    close(f.o_corr[real], ref["o"][rows[real]], "o of the corrupted rows")
    close(f.lse_corr[:, real], ref["lse"][:, rows[real]], "lse of the corrupted rows")
    close(g.dq_clean, ref["dq"][c], "dq of the clean rows")
    close(g.dq_corr[real], ref["dq"][rows[real]], "dq of the corrupted rows")
    close(g.dk_clean, ref["dk"][c], "dk of the clean shard")
    close(g.dv_clean, ref["dv"][c], "dv of the clean shard")
    close(g.dk_corr[real], ref["dk"][rows[real]], "dk of the corrupted keys")
    close(g.dv_corr[real], ref["dv"][rows[real]], "dv of the corrupted keys")


def _rank_worker(rank, world, port, cfg, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, block, H, Hk, d, seed = cfg
        w, x = _inputs(n, block, H, Hk, d, seed)
        plan = csbp.CSBPPlan.build(n, block, world)
        mine = csbp.split_inputs(plan, x.q, x.k, x.v, x.do, rank)
        f, g = csbp.run_rank(plan, mine, OracleOps(w.scale))
        f64 = lambda t: t.numpy()
        ref = oracle.bdlm_attention(f64(x.q), f64(x.k), f64(x.v), block, w.scale, do=f64(x.do))
        _check_rank(plan, rank, x, w, f, g, ref, atol=1e-10)
        out[rank] = "ok"
    except Exception as e:  # reported to the parent
        out[rank] = repr(e)
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,cfg", [(2, (48, 8, 4, 2, 16, 31)), (3, (60, 7, 2, 1, 8, 32)),
                                       (4, (16, 8, 2, 1, 8, 34))])
def test_ranks_exchange_clean_kv_and_their_gradients(world, cfg):
    import torch.multiprocessing as mp

    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_worker, args=(r, world, port, cfg, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert dict(out) == {r: "ok" for r in range(world)}, dict(out)
    assert all(p.exitcode == 0 for p in procs)


def test_all_ranks_in_one_process_match_the_oracle():
    n, block, H, Hk, d = 40, 8, 2, 1, 8
    w, x = _inputs(n, block, H, Hk, d, 33)
    plan = csbp.CSBPPlan.build(n, block, 4)
    xs = [csbp.split_inputs(plan, x.q, x.k, x.v, x.do, r) for r in range(4)]
    outs = csbp.run_local(plan, xs, OracleOps(w.scale))
    f64 = lambda t: t.numpy()
    ref = oracle.bdlm_attention(f64(x.q), f64(x.k), f64(x.v), block, w.scale, do=f64(x.do))
    for r, (f, g) in enumerate(outs):
        _check_rank(plan, r, x, w, f, g, ref, atol=1e-10)


# ----------------------------------------------------------------------------
# the CUDA library, all ranks on one GPU
# ----------------------------------------------------------------------------
@pytest.mark.gpu
@pytest.mark.parametrize("n,block,H,Hk,d,ranks", [(1024, 32, 8, 2, 128, 4), (1200, 16, 4, 2, 64, 3),
                                                  (8192, 64, 8, 2, 128, 8)])
def test_csbp_ranks_on_the_gpu_match_the_oracle(n, block, H, Hk, d, ranks):
    import block_diffusion_lm_bdlm_gb300 as bd

    bd.load_library()
    w = synth.Workload("csbp_gpu", n=n, block=block, heads=H, kv_heads=Hk, head_dim=d, seed=n + ranks, qkv_std=0.5)
    x = synth.make_inputs(w, device="cuda")
    plan = csbp.CSBPPlan.build(n, block, ranks)
    xs = [csbp.split_inputs(plan, x.q, x.k, x.v, x.do, r) for r in range(ranks)]
    outs = csbp.run_local(plan, xs, csbp.GpuOps())
    torch.cuda.synchronize()
    f64 = lambda t: t.double().cpu().numpy()
    ref = oracle.bdlm_attention(f64(x.q), f64(x.k), f64(x.v), block, w.scale, do=f64(x.do))
    from parity_util import check_grad, check_lse, check_o, host

    for r, (f, g) in enumerate(outs):
        p = plan.rank(r)
        rows = np.array(plan.corrupted_rows(r), dtype=np.int64)
        real = rows < 2 * n
        c = slice(p.clean_lo, p.clean_hi)
        check_o(host(f.o_clean), ref["o"][c], f"rank {r} o clean")
        check_lse(host(f.lse_clean), ref["lse"][:, c], f"rank {r} lse clean")
        check_o(host(f.o_corr)[real], ref["o"][rows[real]], f"rank {r} o corrupted")
        check_lse(host(f.lse_corr)[:, real], ref["lse"][:, rows[real]], f"rank {r} lse corrupted")
        check_grad(host(g.dq_clean), ref["dq"][c], f"rank {r} dq clean")
        check_grad(host(g.dq_corr)[real], ref["dq"][rows[real]], f"rank {r} dq corrupted")
        check_grad(host(g.dk_clean), ref["dk"][c], f"rank {r} dk clean shard")
        check_grad(host(g.dv_clean), ref["dv"][c], f"rank {r} dv clean shard")
        check_grad(host(g.dk_corr)[real], ref["dk"][rows[real]], f"rank {r} dk corrupted")
        check_grad(host(g.dv_corr)[real], ref["dv"][rows[real]], f"rank {r} dv corrupted")


def _gather_worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(7)
        full = torch.randn(world * 6, 3, 4, generator=g).to(torch.bfloat16)
        mine = full[rank * 6:(rank + 1) * 6]
        got = csbp._gather_clean(mine)
        assert got.dtype == torch.bfloat16 and torch.equal(got.view(torch.int16), full.view(torch.int16))
        share = torch.randn(world * 6, 2, generator=g) * (rank + 1)
        got_rs = csbp._reduce_scatter_clean(share, rank, world)
        assert got_rs.shape == (6, 2)
        out[rank] = (got_rs.numpy(), share.numpy())
    except Exception as e:
        out[rank] = repr(e)
        raise
    finally:
        dist.destroy_process_group()


def test_gloo_exchange_moves_bf16_bits_and_sums_shares():
    """The all-gather carries bf16 clean K/V bit for bit (as bytes);
    the reduce-scatter leaves each rank the sum of all ranks' shares of its rows."""
    import torch.multiprocessing as mp

    world = 3
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), dict(out)
    shares = [out[r][1] for r in range(world)]
    total = np.sum(shares, axis=0)
    for r in range(world):
        assert np.allclose(out[r][0], total[r * 6:(r + 1) * 6], rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------------------
# two processes, one GPU: gloo ranks whose exchange is staged through host
# memory (their kernels never wait on one another)
# ----------------------------------------------------------------------------
def _local_index(rows_local_to_global, global_rows):
    pos = {int(v): i for i, v in enumerate(rows_local_to_global)}
    return np.array([pos[int(v)] for v in global_rows], dtype=np.int64)


def _check_rank_sampled(plan, rank, x, w, f, g):
    """128K: o, lse, dq of sampled query blocks of this rank (both ends of its
    clean shard, its first and last corrupted blocks) and complete dk, dv of
    its last corrupted key block (and, for the last rank, of the last clean
    key block), on one kv group, against the float64 oracle."""
    from parity_util import check_grad, check_lse, check_o, host

    n, B = w.n, w.block
    G = w.heads // w.kv_heads
    p = plan.rank(rank)
    gk = (3 * rank + 1) % w.kv_heads
    hs = slice(gk * G, (gk + 1) * G)
    q, k, v, do = (t.float().cpu().numpy() for t in (x.q[:, hs], x.k[:, gk:gk + 1], x.v[:, gk:gk + 1], x.do[:, hs]))
    b_lo, b_hi = p.clean_lo // B, p.clean_hi // B
    clean_blocks = [b_lo, b_lo + 1, b_hi - 2, b_hi - 1]
    corr_blocks = [p.blocks[0], p.blocks[-1]]
    row_blocks = [(0, b * B) for b in clean_blocks] + [(0, n + b * B) for b in corr_blocks]
    r = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=row_blocks, want_kv_grads=False)
    crow = np.concatenate([np.arange(b * B, (b + 1) * B) for b in clean_blocks])
    loc = crow - p.clean_lo
    check_o(host(f.o_clean[loc][:, hs]), r["o"][crow], f"rank {rank} o clean")
    check_lse(host(f.lse_clean[hs][:, loc]), r["lse"][:, crow], f"rank {rank} lse clean")
    check_grad(host(g.dq_clean[loc][:, hs]), r["dq"][crow], f"rank {rank} dq clean")
    rows_c = np.array(plan.corrupted_rows(rank), dtype=np.int64)
    xrow = np.concatenate([n + np.arange(b * B, (b + 1) * B) for b in corr_blocks])
    li = _local_index(rows_c, xrow)
    check_o(host(f.o_corr[li][:, hs]), r["o"][xrow], f"rank {rank} o corrupted")
    check_lse(host(f.lse_corr[hs][:, li]), r["lse"][:, xrow], f"rank {rank} lse corrupted")
    check_grad(host(g.dq_corr[li][:, hs]), r["dq"][xrow], f"rank {rank} dq corrupted")
    # complete gradients of one corrupted key block (seen only by its own block)
    b = p.blocks[-1]
    keys = n + np.arange(b * B, (b + 1) * B)
    rk = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=[(0, n + b * B)])
    li = _local_index(rows_c, keys)
    check_grad(host(g.dk_corr[li][:, gk:gk + 1]), rk["dk"][keys], f"rank {rank} dk corrupted block {b}")
    check_grad(host(g.dv_corr[li][:, gk:gk + 1]), rk["dv"][keys], f"rank {rank} dv corrupted block {b}")
    if p.clean_hi == n:  # the last clean key block: seen by its own clean block only
        keys = np.arange(n - B, n)
        rk = oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=[(0, n - B)])
        loc = keys - p.clean_lo
        check_grad(host(g.dk_clean[loc][:, gk:gk + 1]), rk["dk"][keys], f"rank {rank} dk last clean block")
        check_grad(host(g.dv_clean[loc][:, gk:gk + 1]), rk["dv"][keys], f"rank {rank} dv last clean block")


def _gpu_rank_worker(rank, world, port, spec, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import block_diffusion_lm_bdlm_gb300 as bd
        from parity_util import check_grad, check_lse, check_o, host

        bd.load_library()
        if spec[0] == "small":
            _, n, block, H, Hk, d = spec
            w = synth.Workload("csbp_2p", n=n, block=block, heads=H, kv_heads=Hk, head_dim=d, seed=n + 17,
                               qkv_std=0.5)
        else:
            w = synth.BY_NAME[spec[1]]
        x = synth.make_inputs(w, device="cuda")
        plan = csbp.CSBPPlan.build(w.n, w.block, world)
        mine = csbp.split_inputs(plan, x.q, x.k, x.v, x.do, rank)
        f, g = csbp.run_rank(plan, mine, csbp.GpuOps())
        torch.cuda.synchronize()
        if spec[0] == "small":
            f64 = lambda t: t.double().cpu().numpy()
            ref = oracle.bdlm_attention(f64(x.q), f64(x.k), f64(x.v), w.block, w.scale, do=f64(x.do))
            p = plan.rank(rank)
            rows = np.array(plan.corrupted_rows(rank), dtype=np.int64)
            real = rows < 2 * w.n
            c = slice(p.clean_lo, p.clean_hi)
            check_o(host(f.o_clean), ref["o"][c], f"rank {rank} o clean")
            check_lse(host(f.lse_clean), ref["lse"][:, c], f"rank {rank} lse clean")
            check_o(host(f.o_corr)[real], ref["o"][rows[real]], f"rank {rank} o corrupted")
            check_lse(host(f.lse_corr)[:, real], ref["lse"][:, rows[real]], f"rank {rank} lse corrupted")
            check_grad(host(g.dq_clean), ref["dq"][c], f"rank {rank} dq clean")
            check_grad(host(g.dq_corr)[real], ref["dq"][rows[real]], f"rank {rank} dq corrupted")
            check_grad(host(g.dk_clean), ref["dk"][c], f"rank {rank} dk clean shard")
            check_grad(host(g.dv_clean), ref["dv"][c], f"rank {rank} dv clean shard")
            check_grad(host(g.dk_corr)[real], ref["dk"][rows[real]], f"rank {rank} dk corrupted")
            check_grad(host(g.dv_corr)[real], ref["dv"][rows[real]], f"rank {rank} dv corrupted")
        else:
            _check_rank_sampled(plan, rank, x, w, f, g)
        out[rank] = "ok"
    except Exception as e:  # reported to the parent
        out[rank] = repr(e)
        raise
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("spec", [("small", 1024, 32, 8, 2, 128), ("small", 1536, 16, 4, 2, 64),
                                  ("long", "long128k_n131072_b64_h32kv8_d128")])
def test_csbp_two_processes_share_one_gpu(spec):
    """Two ranks as two processes on cuda:0, with gloo moving the clean K/V
    shards and the clean keys' gradient shares through host memory: every
    rank's o, lse, dq and its dk, dv after the reduce-scatter against the
    float64 oracle (in full for the small cases; at 128K on sampled blocks
    and key blocks of one kv group per rank)."""
    import torch.multiprocessing as mp

    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_gpu_rank_worker, args=(r, world, port, spec, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=900)
    for p in procs:
        if p.is_alive():
            p.terminate()
            p.join(timeout=60)
    assert dict(out) == {r: "ok" for r in range(world)}, dict(out)
    assert all(p.exitcode == 0 for p in procs)
