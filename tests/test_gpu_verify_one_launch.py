"""The single-launch verify producer (moe_fp8_verify_produce_one_launch: routing, gate/up, SiLU
and quantisation, down partials and metadata in one launch of 16-CTA clusters; netra-kernel
README, prefill-pair build section) with the route reducer moe_fp8_verify_reduce, behind the
exact batch guard of the verify_m12 profile (12 tokens, h2048 i768 e128 top-8).

Checked here: the routing equals moe_route bit for bit; the activation codes and scales and
the output equal the few-row pair kernels (moe_fp8_gate_up_direct + moe_fp8_down_combine)
bit for bit; everything is inside the oracle contract (ids and hidden codes bit-exact,
activation codes in their window, the output bound given the activation codes); 100
launches are bitwise identical; a CUDA graph replays it; the status word stays clean.
The host-side guard (any other batch or shape refused) is tested on the CPU in
tests/test_abi_host.py.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = [
    pytest.mark.gpu,
    # Kept off the GPU: the producer passed these tests and 20,000-step timed runs, but it
    # failed under a profiler's kernel replay (twice, with and without the teardown drain) and
    # in a timestamp-instrumented copy; until that cause is found by reading, it does not run.
    pytest.mark.skip(reason="verify producer kept off the GPU until the cause of its replay-time faults is found"),
]

if torch.cuda.is_available():
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import GpuMoE, check_act, check_out_given_act, oracle_forward, to_dev, u16

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


def produce_reduce(g, hid_d, renorm=True):
    ids = torch.full((M, g.K), -5, dtype=torch.int32, device="cuda")
    w = torch.full((M, g.K), -5.0, dtype=torch.float32, device="cuda")
    out = torch.empty((M, g.H), dtype=torch.int16, device="cuda")
    L.moe_fp8_verify_produce_one_launch(hid_d, g.router, g.bias, M, renorm, g.w13, g.s13, g.w2, g.s2, ids, w, g.ws, g.shape)
    L.moe_fp8_verify_reduce(w, M, out, g.ws, g.shape)
    return ids, w, out


def pair_views(g):
    a = g.ws_arrays(M)
    return {k: a[k].copy() for k in ("qa", "sa", "act", "act_scale", "row_src", "perm_row")}


CASES = [("verify", True), ("verify_skewed", True), ("verify", False)]


@pytest.mark.parametrize("name,renorm", CASES, ids=[f"{n}-{'renorm' if r else 'full'}" for n, r in CASES])
def test_verify_matches_router_and_pair_kernels(name, renorm):
    x = workload(name)
    g = GpuMoE(x, M)
    g.ws.fill_(0xFF)
    L.moe_fp8_workspace_init(g.ws, g.shape)
    hid_d = to_dev(x.hidden[:M])
    ids, w, out = produce_reduce(g, hid_d, renorm)
    torch.cuda.synchronize()
    assert g.status() == 0
    got = pair_views(g)
    # the same layer through moe_route and the two pair kernels
    ids2, w2 = g.route(hid_d, M, renorm=renorm)
    out2 = torch.empty_like(out)
    L.moe_fp8_gate_up_direct(hid_d, ids2, M, g.w13, g.s13, g.ws, g.shape)
    L.moe_fp8_down_combine(ids2, w2, M, g.w2, g.s2, out2, g.ws, g.shape)
    torch.cuda.synchronize()
    ref = pair_views(g)
    assert torch.equal(ids, ids2) and torch.equal(w, w2)
    for k in ("qa", "sa", "act", "act_scale"):
        assert np.array_equal(got[k], ref[k]), k
    assert torch.equal(out, out2)
    assert np.array_equal(got["perm_row"][:M * g.K], np.arange(M * g.K))
    # the oracle contract
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, x.bias, g.K, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)
    out_o, dbg = oracle_forward(x, x.hidden[:M], ids_o, w_o, debug=True)
    assert np.array_equal(got["qa"], dbg["qa"]) and np.array_equal(got["sa"], dbg["sa"])
    ws = dict(got)
    ws["row_src"] = np.arange(M * g.K, dtype=np.int32)
    check_act(ws, dbg, g.K, f"verify producer {name}")
    check_out_given_act(u16(out), out_o, ws, dbg, ids_o, w_o, x, f"verify producer {name}")


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
    L.moe_fp8_verify_produce_one_launch(to_dev(hidden), g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, ids, w, g.ws, g.shape)
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
    ref = (ids.clone(), w.clone(), out.clone(), pair_views(g)["act"])
    for _ in range(100):
        i2, w2, o2 = produce_reduce(g, hid_d)
        torch.cuda.synchronize()
        assert torch.equal(i2, ref[0]) and torch.equal(w2, ref[1]) and torch.equal(o2, ref[2])
    assert np.array_equal(pair_views(g)["act"], ref[3])
    s = torch.cuda.Stream()
    ids3 = torch.empty_like(ids)
    w3 = torch.empty_like(w)
    out3 = torch.empty_like(out)

    def step():
        L.moe_fp8_verify_produce_one_launch(hid_d, g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, ids3, w3, g.ws, g.shape)
        L.moe_fp8_verify_reduce(w3, M, out3, g.ws, g.shape)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    out3.zero_()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out3, ref[2]) and torch.equal(ids3, ref[0])
    assert g.status() == 0
