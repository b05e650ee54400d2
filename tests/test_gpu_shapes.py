"""GPU parity at the edges of the supported shape set, in both execution modes.

The netra-kernel README's kernel-contract list makes the op's dimensions part of a kernel's
identity and asks for exact guards on them; these cases run the extremes the library
accepts against the CPU oracle: the largest hidden and intermediate sizes (H=8192,
I=4096), the most experts with the largest top-k (E=256, K=16: routing with the
cluster router and the fused combine over 16-CTA clusters), and top-1. Each shape runs
once with few routed rows (one unit per (token, slot) pair) and once with enough rows
for the sorted expert tiles.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import GpuMoE, check_out, oracle_forward, oracle_route, to_dev, u16

EDGE = [("max_dims", 2), ("max_dims", 16), ("many_experts", 2), ("many_experts", 24),
        ("top1", 5), ("top1", 100)]
_CACHE = {}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    import oracle
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()
    yield
    _CACHE.clear()


@pytest.mark.parametrize("name,M", EDGE, ids=[f"{n}-M{m}" for n, m in EDGE])
def test_edge_shape_parity(name, M):
    if name not in _CACHE:
        _CACHE[name] = inputs.make(name)  # the config's M rows; cases take a prefix
    x = _CACHE[name]
    K = x.shape.top_k
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    out = u16(g.forward(hid, ids, w, M))
    torch.cuda.synchronize()
    assert g.status() == 0
    ids_o, w_o = oracle_route(x, rows=slice(0, M))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)
    assert ids_o.shape == (M, K)
    check_out(out, oracle_forward(x, x.hidden[:M], ids_o, w_o), f"{name} M={M}")


ROUTE_WIDE = [(6144, 256, 1), (8192, 256, 1), (8192, 256, 5), (8192, 256, 40), (8192, 128, 3)]


@pytest.mark.parametrize("H,E,M", ROUTE_WIDE, ids=[f"H{h}-E{e}-M{m}" for h, e, m in ROUTE_WIDE])
def test_route_largest_router_matrices(H, E, M):
    """Router matrices too large for a CTA's chunks to sit in shared memory at once (they are
    streamed through it chunk by chunk) against the oracle; the expert FFN is not involved."""
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    K = 8
    hid = inputs.hidden_states(9, M, H)
    wr = inputs.router_weights(9, H, E, 0.02)
    shape = L.make_shape(H, 128, E, K, M)
    ids = torch.empty((M, K), dtype=torch.int32, device="cuda")
    w = torch.empty((M, K), dtype=torch.float32, device="cuda")
    L.moe_route(to_dev(hid), to_dev(wr), None, M, shape, True, ids, w)
    torch.cuda.synchronize()
    ids_o, w_o = oracle.route(hid, wr, None, K)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)
