"""The speculative-verify layer as two operations (netra-kernel README, prefill-pair build
section): moe_fp8_verify_produce (routing, then the quantise-and-sort and the expert-grouped
gate/up, SiLU and requantisation and down kernels, leaving the down partials and the
permutation in the workspace) and moe_fp8_verify_reduce (the route reducer), behind the exact
batch guard of the verify_m12 profile (12 tokens, h2048 i768 e128 top-8).

Checked here: produce + reduce equals moe_fp8_route_forward bit for bit (ids, weights, out and
the workspace's codes); the routing equals the oracle's; everything is inside the oracle
contract (hidden codes bit-exact, the permutation stable and complete, activation codes in
their window, the output bound given the activation codes); zero rows give zero output and
rows past M stay untouched; 100 launches are bitwise identical and a CUDA graph replays them.
The host-side guard (any other batch or shape refused) is tested on the CPU in
tests/test_abi_host.py.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import GpuMoE, check_act, check_out_given_act, check_permutation, oracle_forward, to_dev, u16

M = 12
_CACHE = {}


@pytest.fixture(scope="module", autouse=True)
def _build():
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()
    yield
    _CACHE.clear()


def workload(name):
    if name not in _CACHE:
        _CACHE[name] = inputs.make(name)
    return _CACHE[name]


def produce_reduce(g, hid_d, renorm=True, out=None, ids=None, w=None):
    ids = torch.full((M, g.K), -5, dtype=torch.int32, device="cuda") if ids is None else ids
    w = torch.full((M, g.K), -5.0, dtype=torch.float32, device="cuda") if w is None else w
    out = torch.empty((M, g.H), dtype=torch.int16, device="cuda") if out is None else out
    L.moe_fp8_verify_produce(hid_d, g.router, g.bias, M, renorm, g.w13, g.s13, g.w2, g.s2, ids, w, g.ws, g.shape)
    L.moe_fp8_verify_reduce(w, M, out, g.ws, g.shape)
    return ids, w, out


def views(g):
    a = g.ws_arrays(M)
    return {k: a[k].copy() for k in ("qa", "sa", "act", "act_scale", "row_src", "perm_row", "offsets")}


CASES = [("verify", True), ("verify_skewed", True), ("verify", False)]


@pytest.mark.parametrize("name,renorm", CASES, ids=[f"{n}-{'renorm' if r else 'full'}" for n, r in CASES])
def test_verify_equals_route_forward_and_oracle(name, renorm):
    x = workload(name)
    g = GpuMoE(x, M)
    g.ws.fill_(0xFF)
    L.moe_fp8_workspace_init(g.ws, g.shape)
    hid_d = to_dev(x.hidden[:M])
    ids, w, out = produce_reduce(g, hid_d, renorm)
    torch.cuda.synchronize()
    assert g.status() == 0
    got = views(g)
    # the same layer in one call
    ids2 = torch.empty_like(ids)
    w2 = torch.empty_like(w)
    out2 = torch.empty_like(out)
    L.moe_fp8_route_forward(hid_d, g.router, g.bias, M, renorm, g.w13, g.s13, g.w2, g.s2, out2, ids2, w2, g.ws, g.shape)
    torch.cuda.synchronize()
    ref = views(g)
    assert torch.equal(ids, ids2) and torch.equal(w, w2) and torch.equal(out, out2)
    for k in ("qa", "sa", "act", "act_scale", "perm_row"):
        assert np.array_equal(got[k], ref[k]), k
    # the oracle contract
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, x.bias, g.K, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)
    out_o, dbg = oracle_forward(x, x.hidden[:M], ids_o, w_o, debug=True)
    assert np.array_equal(got["qa"], dbg["qa"]) and np.array_equal(got["sa"], dbg["sa"])
    check_permutation(got, ids_o, g.E)
    check_act(got, dbg, g.K, f"verify producer {name}")
    check_out_given_act(u16(out), out_o, got, dbg, ids_o, w_o, x, f"verify producer {name}")


def test_verify_zero_rows_and_rows_past_m():
    """Zero hidden rows (padding) give exactly zero output; rows >= 12 of the buffers stay
    untouched."""
    x = workload("verify")
    g = GpuMoE(x, 16)
    hidden = x.hidden[:M].copy()
    hidden[[3, 11]] = 0
    ids = torch.full((16, g.K), -777, dtype=torch.int32, device="cuda")
    w = torch.full((16, g.K), -7.0, dtype=torch.float32, device="cuda")
    out = torch.full((16, g.H), -1, dtype=torch.int16, device="cuda")
    L.moe_fp8_verify_produce(to_dev(hidden), g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, ids, w, g.ws, g.shape)
    L.moe_fp8_verify_reduce(w, M, out, g.ws, g.shape)
    torch.cuda.synchronize()
    o = u16(out)
    assert np.all(o[[3, 11]] == 0)
    assert np.all(o[M:] == 0xFFFF) and torch.all(ids[M:] == -777) and torch.all(w[M:] == -7.0)
    ids_o, w_o = oracle.route(hidden, x.router_w, x.bias, g.K)
    assert np.array_equal(ids[:M].cpu().numpy(), ids_o)  # all-zero rows: ties to experts 0..7
    assert g.status() == 0


def test_verify_100_launches_and_graph_replay():
    x = workload("verify_skewed")
    g = GpuMoE(x, M)
    hid_d = to_dev(x.hidden[:M])
    ids, w, out = produce_reduce(g, hid_d)
    torch.cuda.synchronize()
    ref = (ids.clone(), w.clone(), out.clone(), views(g)["act"])
    for _ in range(100):
        i2, w2, o2 = produce_reduce(g, hid_d)
        torch.cuda.synchronize()
        assert torch.equal(i2, ref[0]) and torch.equal(w2, ref[1]) and torch.equal(o2, ref[2])
    assert np.array_equal(views(g)["act"], ref[3])
    s = torch.cuda.Stream()
    ids3 = torch.empty_like(ids)
    w3 = torch.empty_like(w)
    out3 = torch.empty_like(out)
    with torch.cuda.stream(s):
        produce_reduce(g, hid_d, out=out3, ids=ids3, w=w3)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        produce_reduce(g, hid_d, out=out3, ids=ids3, w=w3)
    out3.zero_()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out3, ref[2]) and torch.equal(ids3, ref[0])
    assert g.status() == 0
