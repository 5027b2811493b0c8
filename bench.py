"""Benchmark of the BDLM attention hot path on GB300.

One step = the whole hot path over one synthetic 128K + 128K sequence
(32 query heads / 8 kv heads, head_dim 128, block 64):
  tile enumeration -> 8 partial forwards against contiguous clean-K/V shards
  + 1 partial forward against the local corrupted K/V -> LSE merge of the 9
  partials -> full backward (preprocess, key-major main kernel, dq convert).
Metric: valid-pair TFLOP/s, FLOPs = 4*d*H*P (forward) + 10*d*H*P (backward),
P = n(n + B) valid (query, key) pairs per head.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME]

The other workloads of synth run laid out as they are stated: the 8K + 8K
and packed-document workloads as one forward and one backward, the 256K +
256K workload as its clean rows plus its 16 early/late block groups (see
Step).

Prints one JSON line (rank 0). With --gpus N > 1 (torchrun) every rank runs
an independent replica of the step on its own GPU; the timing is the max over
ranks and the value the FLOPs of all ranks over that time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

WORKLOAD = synth.BY_NAME["long128k_n131072_b64_h32kv8_d128"]
METRIC = "BDLM attn fwd+bwd TFLOP/s (valid pairs) and % BF16 peak at 128K, 1 GB300"
UNIT = "TFLOP/s"

# dram traffic of the dominant kernel per launch from an ncu capture, valid
# while the sources it is compiled from are unchanged (checked by hash;
# otherwise reported as null)
TRAFFIC = {"kernel_sources": ['block_diffusion_lm_bdlm_gb300/csrc/bwd_tc.cu', 'block_diffusion_lm_bdlm_gb300/csrc/common.cuh', 'block_diffusion_lm_bdlm_gb300/csrc/tc_ptx.cuh', 'block_diffusion_lm_bdlm_gb300/csrc/kernels.h'],
           "sha1": "25840ed9639536ee7e102deddc0538139b1a0c85",
           "bytes_per_launch": 107317465088 + 62680961792,
           "note": "bwd_tc_kernel on this workload, ncu dram__bytes_read.sum + dram__bytes_write.sum"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def valid_pairs(n, block):
    """Valid (query, key) pairs per head of one sequence of clean length n:
    n (n + B) when B divides n; with n = nb B + r, B^2 nb (nb + 1) + 2 r n."""
    nb, r = divmod(n, block)
    return block * block * nb * (nb + 1) + 2 * r * n


def step_flops(w):
    if w.docs:  # packed documents: each document is [clean n_d | corrupted n_d]
        P = sum(valid_pairs(ln // 2, w.block) for ln in synth.doc_lengths(w))
    else:
        P = valid_pairs(w.n, w.block)
    return 4 * w.head_dim * w.heads * P, 10 * w.head_dim * w.heads * P


def merge_bytes(w, n_parts):
    if n_parts == 0:
        return 0
    rows, per = 2 * w.n, w.heads
    unit = 2 * w.head_dim + 4  # bf16 row of o + fp32 lse
    return rows * per * unit * (n_parts + 1)


def mufu_exp_peak(clocks):
    """Exponentials per second the special-function units can issue, times
    the SM count, at the median SM clock sampled under load (the maximum
    clock when no sample): 32 ex2 per clock per SM on compute capability 10.3
    (GB300 doubles the exponential rate of the sm_100 parts, 16 per clock per
    SM; a timing probe of ex2.approx.ftz.f32 with one packed FMA per pair, two
    warps per SM sub-partition on all SMs, measured about 29 per clock)."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    per_clk = 32.0 if (props.major, props.minor) == (10, 3) else 16.0
    mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070
    return per_clk * props.multi_processor_count * float(mhz) * 1e6


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    # raw samples go to BDLM_CLOCKS_DIR (default: the system temporary
    # directory); the JSON line carries their summary
    def __init__(self, index, tag="timed"):
        self.index = index
        self.proc = None
        d = os.environ.get("BDLM_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_{tag}_gpu{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception as e:  # pragma: no cover
            log("clock sampling unavailable:", e)
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "sm_mhz_min": min(sm) if sm else None, "power_w_median": statistics.median(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_sha(rels):
    h = hashlib.sha1()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------------------------
# the oracle leg (CPU baseline / reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(x_host, w, budget_s):
    """Run the float64 oracle (forward + backward) on query blocks of kv group
    0 of the workload, latest blocks first (the heaviest rows), until budget_s
    of CPU time is spent. Returns (valid pairs per second, pairs, seconds, blocks)."""
    import numpy as np

    import oracle

    G = w.heads // w.kv_heads
    q, k, v, do = x_host
    n, B = w.n, w.block
    nb = n // B
    order = []
    for b in range(nb - 1, -1, -1):
        order += [(0, b * B), (0, n + b * B)]
    t0 = time.perf_counter()
    pairs = 0
    done = 0
    for blk in order:
        oracle.bdlm_attention(q, k, v, B, w.scale, do=do, row_blocks=[blk])
        b = (blk[1] % n) // B
        pairs += B * (b + 1) * B * G
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return pairs / dt, pairs, dt, done


def host_group0(x, w):
    import numpy as np

    G = w.heads // w.kv_heads
    f = lambda t: t.float().cpu().numpy()
    return (f(x.q[:, :G]), f(x.k[:, :1]), f(x.v[:, :1]), f(x.do[:, :G]))


def oracle_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w = WORKLOAD
    # one kv group of the workload (G query heads, 1 kv head), same shapes and
    # distributions, drawn on the CPU
    G = w.heads // w.kv_heads
    wg = synth.Workload(w.name + "_group0", n=w.n, block=w.block, heads=G, kv_heads=1, head_dim=w.head_dim,
                        seed=w.seed, qkv_std=w.qkv_std)
    x = synth.make_inputs(wg, device="cpu")
    xh = host_group0(x, wg)
    flop_per_pair = 14 * w.head_dim
    for _ in range(args.warmup):
        oracle_sample(xh, w, budget_s=0.5)
    times, pairs = [], []
    for _ in range(args.steps):
        rate, pr, dt, nblk = oracle_sample(xh, w, budget_s=args.ref_budget)
        times.append(dt)
        pairs.append(pr)
    total_pairs, total_t = sum(pairs), sum(times)
    value = flop_per_pair * total_pairs / total_t / 1e12
    sample = (f"float64 oracle fwd+bwd on the latest query blocks (B={w.block} rows each, kv group 0 = "
              f"{w.heads // w.kv_heads} q heads) of the 128K workload, ~{args.ref_budget:.0f} s per step")
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_pairs_per_step": total_pairs // args.steps},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------
# the CUDA arm
# ----------------------------------------------------------------------------
class Step:
    """One pass of the hot path over one batch, laid out as the workload
    states it:
      shards  the partial forwards against the contiguous clean-K/V shards
              and the local corrupted keys, their LSE merge, the backward;
      full    one forward and one backward over the sequence, or over the
              packed documents (cu_seqlens);
      groups  block parallelism: the clean rows' forward against the clean
              keys, then every early/late block group's forward (its
              corrupted rows against all clean keys and its own corrupted
              keys), then the same backwards. The groups' shares of the clean
              keys' dk, dv stay per group, as on the ranks that own them (their
              sum is a multi-GPU reduction, out of scope on one GPU); each
              group's inputs are laid out once, before any timing, as a
              rank would hold them."""

    def __init__(self, bd, w, x, dev):
        self.bd, self.w, self.x = bd, w, x
        H, d = w.heads, w.head_dim
        self.cu = None
        self.mode = "full" if w.docs else ("shards" if w.shards else ("groups" if w.groups else "full"))
        self.windows = []
        if w.docs:
            self.cu = torch.tensor(x.cu_seqlens, dtype=torch.int32, device=dev)
            L, n_docs = x.cu_seqlens[-1], w.docs
        else:
            n = w.n
            L, n_docs = 2 * n, 1
            if self.mode == "shards":
                self.windows = synth.shard_bounds(n, w.shards) + [(n, 2 * n)]
        self.groups = self._layout_groups(dev) if self.mode == "groups" else []
        # the partials as one [P, L, H, d] buffer (and [P, H, L] lse): the
        # window calls write its slices, a task list writes its slots
        P = len(self.windows)
        self.parts_all = torch.empty((P,) + tuple(x.q.shape), dtype=x.q.dtype, device=dev) if P else None
        self.plse_all = torch.empty((P, H, L), dtype=torch.float32, device=dev) if P else None
        self.parts = [self.parts_all[i] for i in range(P)]
        self.plse = [self.plse_all[i] for i in range(P)]
        self.tasks = [bd.Task(0, w.n, 0, 2 * w.n, lo, hi, i) for i, (lo, hi) in enumerate(self.windows)]
        self.ws_t = torch.empty(max(bd.bdlm_attn_fwd_tasks_workspace_bytes(self.tasks), 256), dtype=torch.uint8,
                                device=dev) if P else None
        self.o = torch.empty_like(x.q)
        self.lse = torch.empty((H, L), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(x.q)
        self.dk = torch.empty_like(x.k)
        self.dv = torch.empty_like(x.v)
        self.ws_f = torch.empty(bd.bdlm_attn_fwd_workspace_bytes(L, H, d, n_docs), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(bd.bdlm_attn_bwd_workspace_bytes(L, H, d, n_docs), dtype=torch.uint8, device=dev)
        self.launches = 0

    def _layout_groups(self, dev):
        """Per group: its block list and its gathered q, k, v, dO (q, dO: the
        corrupted rows of its blocks; k, v: the n clean rows, then those rows),
        with its outputs; plus the clean rows (views of the inputs)."""
        w, x = self.w, self.x
        n, B, H = w.n, w.block, w.heads
        ar = torch.arange(B, device=dev)
        clean = torch.arange(n, device=dev)
        gs = []
        for blocks in synth.early_late_groups((n + B - 1) // B, w.groups):
            bl = torch.tensor(blocks, dtype=torch.int32, device=dev)
            corr = (n + bl.long()[:, None] * B + ar[None]).reshape(-1)
            kpos = torch.cat([clean, corr])
            g = dict(bl=bl, q=x.q[corr].contiguous(), k=x.k[kpos].contiguous(), v=x.v[kpos].contiguous(),
                     do=x.do[corr].contiguous())
            g["o"] = torch.empty_like(g["q"])
            g["lse"] = torch.empty((H, g["q"].shape[0]), dtype=torch.float32, device=dev)
            g["dq"], g["dk"], g["dv"] = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
            gs.append(g)
        c = dict(q=x.q[:n], k=x.k[:n], v=x.v[:n], do=x.do[:n], o=torch.empty_like(x.q[:n]),
                 lse=torch.empty((H, n), dtype=torch.float32, device=dev), dq=torch.empty_like(x.q[:n]),
                 dk=torch.empty_like(x.k[:n]), dv=torch.empty_like(x.v[:n]))
        self.clean = c
        return gs

    def _groups_fwd(self):
        bd, w = self.bd, self.w
        n, B, c = w.n, w.block, self.clean
        launches = 0
        bd.bdlm_attn_fwd(c["q"], c["k"], c["v"], B, L=2 * n, part=bd.Partial.window(0, n, q_lo=0, q_hi=n),
                         out=c["o"], lse=c["lse"], workspace=self.ws_f)
        launches += bd.bdlm_last_launch_count()
        for g in self.groups:
            bd.bdlm_attn_fwd(g["q"], g["k"], g["v"], B, L=2 * n, part=bd.Partial.group(g["bl"]), out=g["o"],
                             lse=g["lse"], workspace=self.ws_f)
            launches += bd.bdlm_last_launch_count()
        return launches

    def _groups_bwd(self):
        bd, w = self.bd, self.w
        n, B, c = w.n, w.block, self.clean
        launches = 0
        bd.bdlm_attn_bwd(c["q"], c["k"], c["v"], c["o"], c["lse"], c["do"], B, L=2 * n,
                         part=bd.Partial.window(0, n, q_lo=0, q_hi=n), dq=c["dq"], dk=c["dk"], dv=c["dv"],
                         workspace=self.ws_b)
        launches += bd.bdlm_last_launch_count()
        for g in self.groups:
            bd.bdlm_attn_bwd(g["q"], g["k"], g["v"], g["o"], g["lse"], g["do"], B, L=2 * n,
                             part=bd.Partial.group(g["bl"]), dq=g["dq"], dk=g["dk"], dv=g["dv"], workspace=self.ws_b)
            launches += bd.bdlm_last_launch_count()
        return launches

    def run(self, ev=None, after_fwd=None):
        """One step; `after_fwd` (if given) is called between the forward
        (with its merge) and the backward."""
        bd, w, x = self.bd, self.w, self.x
        launches = 0
        if ev:
            ev[0].record()
        for (lo, hi), po, pl in zip(self.windows, self.parts, self.plse):
            bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], w.block, part=bd.Partial.window(lo, hi), out=po, lse=pl,
                             workspace=self.ws_f)
            launches += bd.bdlm_last_launch_count()
        if self.mode == "full":
            bd.bdlm_attn_fwd(x.q, x.k, x.v, w.block, cu_seqlens=self.cu, out=self.o, lse=self.lse, workspace=self.ws_f)
            launches += bd.bdlm_last_launch_count()
        elif self.mode == "groups":
            launches += self._groups_fwd()
        if ev:
            ev[1].record()
        if self.windows:
            bd.bdlm_lse_merge(self.parts, self.plse, out=self.o, lse=self.lse)
            launches += bd.bdlm_last_launch_count()
        if ev:
            ev[2].record()
        if after_fwd:
            after_fwd()
        if self.mode == "groups":
            launches += self._groups_bwd()
        else:
            bd.bdlm_attn_bwd(x.q, x.k, x.v, self.o, self.lse, x.do, w.block, cu_seqlens=self.cu, dq=self.dq,
                             dk=self.dk, dv=self.dv, workspace=self.ws_b)
            launches += bd.bdlm_last_launch_count()
        if ev:
            ev[3].record()
        self.launches += launches

    def time_task_list(self, reps=3):
        """The same partial forwards as one task list (one attention launch
        over all windows, into the same partial buffers), and the backward of
        the same windows as one task list (each window's keys complete, dq
        summed over the windows: the full backward, key window by key window);
        not part of the timed step. Returns the median ms of `reps` runs after
        one warm-up of each (None, None for packed documents)."""
        bd, w, x = self.bd, self.w, self.x
        if not self.windows:
            return None, None
        bwd_tasks = [bd.Task(0, w.n, 0, 2 * w.n, lo, hi, 0) for lo, hi in self.windows]
        L, H, d = x.q.shape
        ws_b = torch.empty(bd.bdlm_attn_bwd_tasks_workspace_bytes(bwd_tasks, L, H, d), dtype=torch.uint8,
                           device=x.q.device)

        def fwd():
            bd.bdlm_attn_fwd_tasks(x.q, x.k, x.v, w.block, self.tasks, len(self.tasks), out=self.parts_all,
                                   lse=self.plse_all, workspace=self.ws_t)

        def bwd():
            bd.bdlm_attn_bwd_tasks(x.q, x.k, x.v, self.o, self.lse, x.do, w.block, bwd_tasks, 1, dq=self.dq,
                                   dk=self.dk.unsqueeze(0), dv=self.dv.unsqueeze(0), workspace=ws_b)

        out = []
        for f in (fwd, bwd):
            f()
            times = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                f()
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            out.append(statistics.median(times))
        del ws_b
        return out[0], out[1]

    def time_graph(self, reps=5):
        """The step captured once in a CUDA graph and replayed (every library
        call only launches kernels on the current stream, with all host-side
        values in kernel parameters). Returns the median ms per replay after
        one warm-up replay; not part of the timed step."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        g.replay()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        del g
        return statistics.median(times)

    def time_running_merge(self, reps=2):
        """The same windows merged by the forward's epilogue into a running
        fp32 (o, lse) instead of kept as partials and merged (not part of the
        timed step). Returns the median ms of `reps` runs after one warm-up
        (None for packed documents, which have no windows)."""
        bd, w, x = self.bd, self.w, self.x
        if not self.windows:
            return None
        ro = torch.empty(x.q.shape, dtype=torch.float32, device=x.q.device)
        rl = torch.empty_like(self.lse)

        def run():
            for i, (lo, hi) in enumerate(self.windows):
                bd.bdlm_attn_fwd(x.q, x.k[lo:hi], x.v[lo:hi], w.block, part=bd.Partial.window(lo, hi, accumulate=i > 0),
                                 out=ro, lse=rl, workspace=self.ws_f)

        run()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        del ro, rl
        return statistics.median(times)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world, dev):
    if world > 1:
        import torch.distributed as dist

        if dev.type == "cuda":
            dist.barrier(device_ids=[dev.index])
        else:
            dist.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_cuda(args, rank, world, local):
    import block_diffusion_lm_bdlm_gb300 as bd

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA arm has no CPU fallback)")
    bd.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.BY_NAME[args.workload]
    log(f"[rank {rank}] generating inputs for {w.name}")
    x = synth.make_inputs(w, device="cuda")
    step = Step(bd, w, x, dev)
    f_fwd, f_bwd = step_flops(w)
    flops = f_fwd + f_bwd

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    step.launches = 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    barrier(world, dev)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for k in range(args.steps):
        step.run(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    barrier(world, dev)
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    launches = step.launches
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    mrg_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    bwd_ms = statistics.median(e[2].elapsed_time(e[3]) for e in evs)
    bwd_mean_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / len(evs)
    step_ms = sorted(e[0].elapsed_time(e[3]) for e in evs)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = flops * world * args.steps / (total_ms / 1e3) / 1e12

    peaks, peak_kind = load_peaks()
    achieved = f_bwd / (bwd_mean_ms / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    run_ms = step.time_running_merge()
    task_ms, task_bwd_ms = step.time_task_list()
    graph_ms = step.time_graph()
    e2e = None
    if not args.no_e2e and step.mode != "groups":
        e2e = end_to_end(step, x, flops, args, world, dev)
    _report(args, rank, world, w, step, x, flops, f_fwd, f_bwd, total_ms, ms_per_step, value, fwd_ms, mrg_ms,
            bwd_ms, achieved, peak, peak_kind, peaks, e2e, launches, clocks, run_ms, step_ms, task_ms,
            task_bwd_ms, graph_ms)


def end_to_end(step, x, flops, args, world, dev):
    """The same step through the public API with host buffers, run as a
    training loop would run it: two device buffer sets, and a copy stream that
    brings step k+1's inputs in from pinned host memory while step k computes
    and takes step k's results out to pinned host memory while step k+1
    computes. Every step's inputs are copied in and every step's results
    copied out inside the timed region. Only the head and the tail are not
    hidden behind compute: step 0's q, k, v (its dO arrives during its
    forward) and the last step's dq, dk, dv (its o and lse leave during its
    backward)."""
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h_in = [pin(t) for t in (x.q, x.k, x.v, x.do)]
    for h, t in zip(h_in, (x.q, x.k, x.v, x.do)):
        h.copy_(t)
    x_b = synth.Inputs(q=torch.empty_like(x.q), k=torch.empty_like(x.k), v=torch.empty_like(x.v),
                       do=torch.empty_like(x.do), cu_seqlens=x.cu_seqlens)
    steps = [step, Step(step.bd, step.w, x_b, dev)]
    ins = lambda st: (st.x.q, st.x.k, st.x.v, st.x.do)
    outs = lambda st: (st.o, st.lse, st.dq, st.dk, st.dv)
    h_out = [pin(t) for t in outs(step)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    comp = torch.cuda.current_stream(dev)
    cs = torch.cuda.Stream(dev)
    Ev = lambda: torch.cuda.Event(enable_timing=True)

    def pipeline(K):
        t0, t1 = Ev(), Ev()
        ev_in = [Ev() for _ in range(K)]    # q, k, v of step k are on the device
        ev_do = [Ev() for _ in range(K)]    # dO of step k is on the device
        ev_fwd = [Ev() for _ in range(K)]   # step k's o, lse are final (forward and merge done)
        ev_done = [Ev() for _ in range(K)]  # step k computed

        def copy_in(k):  # on the copy stream: q, k, v first (the forward needs them), then dO
            dst = ins(steps[k % 2])
            for h, t in zip(h_in[:3], dst[:3]):
                t.copy_(h, non_blocking=True)
            ev_in[k].record(cs)
            dst[3].copy_(h_in[3], non_blocking=True)
            ev_do[k].record(cs)

        t0.record(comp)
        cs.wait_event(t0)
        with torch.cuda.stream(cs):
            copy_in(0)
        for k in range(K):
            st = steps[k % 2]
            comp.wait_event(ev_in[k])

            def between(k=k):  # o, lse can go out now; the backward needs dO
                ev_fwd[k].record(comp)
                comp.wait_event(ev_do[k])

            st.run(after_fwd=between)
            ev_done[k].record(comp)
            with torch.cuda.stream(cs):
                if k + 1 < K:
                    # the other buffer set was last read by step k - 1; its
                    # results went out before this copy (same stream)
                    if k >= 1:
                        cs.wait_event(ev_done[k - 1])
                    copy_in(k + 1)
                res = outs(st)
                cs.wait_event(ev_fwd[k])
                for h, t in zip(h_out[:2], res[:2]):  # o, lse during the backward
                    h.copy_(t, non_blocking=True)
                cs.wait_event(ev_done[k])
                for h, t in zip(h_out[2:], res[2:]):  # dq, dk, dv
                    h.copy_(t, non_blocking=True)
        comp.wait_stream(cs)
        t1.record(comp)
        return t0, ev_in, ev_done, t1

    pipeline(2)  # untimed: the first use of freshly pinned host buffers is slow
    torch.cuda.synchronize()
    e2e_steps = max(1, args.steps)
    sampler = ClockSampler(dev.index, tag="e2e")
    sampler.start()
    barrier(world, dev)
    t0, ev_in, ev_done, t1 = pipeline(e2e_steps)
    torch.cuda.synchronize()
    barrier(world, dev)
    clocks = sampler.stop()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    e2e_value = flops * world * e2e_steps / (e2e_ms / 1e3) / 1e12
    marks = [t0] + ev_done
    del steps[1], x_b
    return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps, "total_ms": e2e_ms,
            "compute_done_ms": [marks[i].elapsed_time(marks[i + 1]) for i in range(e2e_steps)],
            # the exposed head: step 0's inputs arriving, then step 0's compute
            "first_copy_in_ms": t0.elapsed_time(ev_in[0]), "first_step_ms": ev_in[0].elapsed_time(ev_done[0]),
            "overlap": "copy stream; inputs of step k+1 in and results of step k out during compute; "
                       "dO arrives during the forward, o and lse leave during the backward",
            "clocks": clocks}


def l2_note(x):
    qb = x.q.numel() * x.q.element_size()
    if qb > 129e6:
        return f"inputs larger than L2 (q alone {qb / 1e9:.2f} GB > 129 MB L2), no flush"
    return f"inputs smaller than L2 (q {qb / 1e6:.0f} MB): profiling case, not a bench line"


def _report(args, rank, world, w, step, x, flops, f_fwd, f_bwd, total_ms, ms_per_step, value, fwd_ms, mrg_ms,
            bwd_ms, achieved, peak, peak_kind, peaks, e2e, launches, clocks, run_ms, step_ms, task_ms, task_bwd_ms,
            graph_ms=None):
    traffic = None
    if TRAFFIC["sha1"] and source_sha(TRAFFIC["kernel_sources"]) == TRAFFIC["sha1"]:
        traffic = TRAFFIC["bytes_per_launch"]
    mbytes = merge_bytes(w, len(step.windows))
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "n_clean": w.n, "n_corrupted": w.n, "docs": w.docs or 1,
                   "rows": x.q.shape[0], "block": w.block, "heads": w.heads,
                   "kv_heads": w.kv_heads, "head_dim": w.head_dim, "layout": step.mode, "clean_shards": w.shards,
                   "block_groups": w.groups,
                   "l2": l2_note(x), "parallelism": f"replicas{world}"},
        "roofline": {"kernel": "bdlm_attn_bwd (key-major main kernel + preprocess + dq convert)",
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} bf16_tflops_sustained"},
        "components": {
            "fwd_partials_ms": fwd_ms, "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12,
            "merge_ms": mrg_ms if mbytes else None,
            "merge_gbs": mbytes / (mrg_ms / 1e3) / 1e9 if mbytes else None,
            "merge_frac_hbm": mbytes / (mrg_ms / 1e3) / 1e9 / float(peaks["hbm_gbs"]) if mbytes else None,
            "bwd_ms": bwd_ms, "bwd_tflops": f_bwd / (bwd_ms / 1e3) / 1e12,
            "fwd_frac_bf16": f_fwd / (fwd_ms / 1e3) / 1e12 / float(peaks["bf16_tflops"]),
            "bwd_frac_bf16": f_bwd / (bwd_ms / 1e3) / 1e12 / float(peaks["bf16_tflops"]),
            "flops_fwd": f_fwd, "flops_bwd": f_bwd, "merge_bytes": mbytes,
            "fwd_running_merge_ms": run_ms,
            "fwd_running_merge_tflops": f_fwd / (run_ms / 1e3) / 1e12 if run_ms else None,
            "fwd_task_list_ms": task_ms,
            "fwd_task_list_tflops": f_fwd / (task_ms / 1e3) / 1e12 if task_ms else None,
            "bwd_task_list_ms": task_bwd_ms,
            "bwd_task_list_tflops": f_bwd / (task_bwd_ms / 1e3) / 1e12 if task_bwd_ms else None,
            "step_ms_min": step_ms[0], "step_ms_median": statistics.median(step_ms), "step_ms_max": step_ms[-1],
            # the same step replayed from a CUDA graph (outside the timed steps)
            "step_graph_ms": graph_ms,
            "step_graph_tflops": flops / (graph_ms / 1e3) / 1e12 if graph_ms else None,
            # the forward's secondary bound: one exponential per valid (row, key) pair and head
            "fwd_exp_per_s": f_fwd / (4 * w.head_dim) / (fwd_ms / 1e3),
            "fwd_exp_frac_mufu": (f_fwd / (4 * w.head_dim) / (fwd_ms / 1e3)) / mufu_exp_peak(clocks),
        },
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not w.docs:
        xh = host_group0(x, w)
        rate, pr, dt, nblk = oracle_sample(xh, w, budget_s=args.cpu_budget)
        out["cpu_baseline"] = {
            "value": 14 * w.head_dim * rate / 1e12, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"float64 oracle fwd+bwd on {nblk} query blocks (B={w.block} rows, latest first) of kv "
                      f"group 0 ({w.heads // w.kv_heads} q heads) of this workload, {pr} valid pairs in {dt:.1f} s",
        }
    if rank == 0:
        print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--workload", default=WORKLOAD.name,
                    help="workload name from synth (default: the 128K workload; others are for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        log("bench.py: at least 3 warm-up steps are required; using 3")
        args.warmup = 3
    rank, world, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_cuda(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
