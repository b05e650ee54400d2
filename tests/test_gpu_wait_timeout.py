"""The bounded device wait, made to run out on purpose without faulting or hanging the GPU.

Every kernel of the library waits on its own copies, MMAs and cluster peers with a time
limit, and reports a wait that ran out as MOE_STATUS_WAIT_TIMEOUT instead of spinning on.
moe_fp8_selftest_wait waits with that same helper on a barrier phase that nothing will ever
complete (no copy or MMA is issued, so nothing is left in flight), with a limit of
microseconds. The kernel must return, the status bit must be set, and the context must stay
usable: a normal call right after is clean and matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import GpuMoE, check_out, oracle_forward, oracle_route, to_dev, u16


@pytest.fixture(scope="module", autouse=True)
def _build():
    import oracle
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()


def test_wait_runs_out_reports_and_the_context_stays_usable():
    from fp8_block_scaled_router_gb300 import _lib as L
    x = inputs.make("tiny")
    M = 4
    g = GpuMoE(x, M)
    assert g.status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    L.moe_fp8_selftest_wait(g.ws, g.shape, 20)  # give up after 20 us
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert g.status() & L.STATUS_WAIT_TIMEOUT
    assert dt < 5.0
    # cleared by re-initialising the workspace; the next layer call is clean and correct
    L.moe_fp8_workspace_init(g.ws, g.shape)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    out = u16(g.forward(hid, ids, w, M))
    assert g.status() == 0
    ids_o, w_o = oracle_route(x, rows=slice(0, M))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    check_out(out, oracle_forward(x, x.hidden[:M], ids_o, w_o), "after a timed-out wait")


def test_selftest_rejects_out_of_range_limits():
    from fp8_block_scaled_router_gb300 import _lib as L
    x = inputs.make("tiny")
    g = GpuMoE(x, 4)
    assert L.moe_fp8_selftest_wait(g.ws, g.shape, 0, check=False) == 1
    assert L.moe_fp8_selftest_wait(g.ws, g.shape, 2_000_000, check=False) == 1
    assert g.status() == 0
