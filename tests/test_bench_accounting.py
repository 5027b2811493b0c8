"""The benchmark's work accounting against the oracle's mask: the valid-pair
FLOP counts of every workload and the merge's algorithmic bytes (no GPU)."""
import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


@pytest.mark.parametrize("n,block", [(64, 8), (62, 8), (100, 16), (5, 8), (37, 64), (129, 128), (300, 200)])
def test_valid_pairs_count_the_mask(bench, n, block):
    assert bench.valid_pairs(n, block) == int(oracle.full_mask(n, block).sum()) == oracle.valid_pairs(n, block)


def test_step_flops_of_every_workload(bench):
    for w in synth.WORKLOADS:
        f_fwd, f_bwd = bench.step_flops(w)
        if w.docs:
            P = sum(oracle.valid_pairs(ln // 2, w.block) for ln in synth.doc_lengths(w))
        else:
            P = oracle.valid_pairs(w.n, w.block)
        assert f_fwd == 4 * w.head_dim * w.heads * P
        assert f_bwd == 10 * w.head_dim * w.heads * P
    # the headline workload: 2.816e14 + 7.040e14 FLOP per step
    f_fwd, f_bwd = bench.step_flops(bench.WORKLOAD)
    assert abs(f_fwd - 2.816e14) / 2.816e14 < 1e-3 and abs(f_bwd - 7.040e14) / 7.040e14 < 1e-3


def test_merge_bytes_of_the_headline_workload(bench):
    # 9 bf16 partials read and one result written, each row a bf16 o row per
    # head plus its fp32 lse: 19.63 GB read + 2.18 GB written
    w = bench.WORKLOAD
    b = bench.merge_bytes(w, 9)
    per = 2 * w.n * w.heads * (2 * w.head_dim + 4)
    assert b == 10 * per
    assert abs(b / 1e9 - 21.81) < 0.01
    assert bench.merge_bytes(w, 0) == 0


def test_block_group_pairs_cover_the_corrupted_half(bench):
    # the groups' valid pairs (each corrupted row of block b sees b*B clean
    # keys and its B own keys) add up to the corrupted half's share of the mask
    n, block = 96, 8
    m = oracle.full_mask(n, block)
    nb = n // block
    pairs = sum(block * (b * block + block) for g in synth.early_late_groups(nb, 4) for b in g)
    assert pairs == int(m[n:].sum())
    assert np.all(m[:n, n:] == 0)
