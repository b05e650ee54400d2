"""GPU parity at the edges of the supported shape set, in both execution modes.

The netra-kernel README's kernel-contract list makes the op's dimensions part of a kernel's
identity and asks for exact guards on them; these cases run the extremes the library
accepts against the CPU oracle: the largest hidden and intermediate sizes (H=8192,
I=4096), the most experts with the largest top-k (E=256, K=16: routing with the
cluster router and the fused combine over 16-CTA clusters), and top-1. Each shape runs
once with few routed rows (one unit per (token, slot) pair) and once with enough rows
for the sorted expert tiles; top-1 also runs at the borders between the three modes (64/65
routed rows: pairs and expert groups; 256/257: expert groups and sorted tiles), and the most
experts once in the expert-grouped mode (160 routed rows over 256 experts).
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import GpuMoE, check_out, oracle_forward, oracle_route, to_dev, u16

EDGE = [("max_dims", 2), ("max_dims", 16), ("many_experts", 2), ("many_experts", 10), ("many_experts", 24),
        ("top1", 5), ("top1", 64), ("top1", 65), ("top1", 100), ("top1", 256), ("top1", 257)]
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
    key = (name, max(M, inputs.CONFIGS[name]["M"]))
    if key not in _CACHE:
        _CACHE[key] = inputs.make(name, M=key[1])  # cases take a prefix of the rows
    x = _CACHE[key]
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


ROUTE_MANY = [(2048, 128, 4096, True, True), (2048, 128, 777, False, True), (1024, 64, 1000, True, False),
              (4096, 32, 515, True, True), (256, 64, 640, False, False)]


@pytest.mark.parametrize("H,E,M,renorm,with_bias", ROUTE_MANY,
                         ids=[f"H{h}-E{e}-M{m}-{'renorm' if r else 'full'}{'-bias' if b else ''}"
                              for h, e, m, r, b in ROUTE_MANY])
def test_route_many_tokens(H, E, M, renorm, with_bias):
    """The many-token router (32 tokens per CTA) against the oracle: every expert count it
    serves, token counts that leave a partial last block, with and without a bias and
    renormalisation."""
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    K = 8
    hid = inputs.hidden_states(11, M, H)
    wr = inputs.router_weights(11, H, E, 1.0 / np.sqrt(H))
    bias = (np.random.default_rng(11).standard_normal(E) * 0.5).astype(np.float32) if with_bias else None
    shape = L.make_shape(H, 128, E, K, M)
    ids = torch.full((M, K), -3, dtype=torch.int32, device="cuda")
    w = torch.empty((M, K), dtype=torch.float32, device="cuda")
    L.moe_route(to_dev(hid), to_dev(wr), None if bias is None else torch.from_numpy(bias).cuda(), M, shape, renorm,
                ids, w)
    torch.cuda.synchronize()
    ids_o, w_o = oracle.route(hid, wr, bias, K, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)
