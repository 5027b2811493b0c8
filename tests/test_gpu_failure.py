"""The device failure path on the GPU without a fault: a bounded wait that
nothing completes gives up, records BDLM_ERR_TIMEOUT in the workspace, and
the context stays usable for the next call."""
import time

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    import block_diffusion_lm_bdlm_gb300 as m

    m.load_library()
    return m


def test_wait_timeout_is_reported_and_context_survives(bd):
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bd.bdlm_selftest_timeout(ws, wait_ns=50_000_000)
    assert bd.bdlm_read_error(ws) == 5  # BDLM_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.045  # it waited out its limit
    # the same context and workspace run an ordinary call afterwards
    w = synth.Workload("case", n=128, block=16, heads=2, kv_heads=1, head_dim=128, seed=3, qkv_std=0.5)
    x = synth.make_inputs(w, device="cuda")
    o, lse = bd.bdlm_attn_fwd(x.q, x.k, x.v, w.block, workspace=ws)
    assert bd.bdlm_read_error(ws) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
