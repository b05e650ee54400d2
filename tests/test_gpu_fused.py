"""The single-launch layer (moe_fp8_route_forward_one_launch) and the two-call form
(moe_fp8_route_forward).

For up to 16 routed pairs the library can run the whole layer -- routing, the hidden
quantisation, gate/up, SiLU*up with the requantisation, down and the slot-order combine --
as one kernel: the producer stages and the route reducer of the netra-kernel README's
prefill-pair section in one launch. Its routing must be bit-identical to moe_route, its
output bit-identical to moe_route + moe_fp8_forward (= moe_fp8_route_forward), and both within
the oracle contract (ids bit-exact, hidden codes bit-exact, activation codes in their window,
the output bound given the activation codes); its arrival counters must be left at zero after
every call, and rows past M untouched. Shapes outside its limits are refused.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import (GpuMoE, check_act, check_out_given_act, oracle_forward, oracle_route, to_dev,
                             u16)

_CACHE = {}


def workload(name, M):
    key = (name, M)
    if key not in _CACHE:
        _CACHE[key] = inputs.make(name, tokens=max(M, 4)) if name == "decode" else inputs.make(name, M=max(M, 4))
    return _CACHE[key]


@pytest.fixture(scope="module", autouse=True)
def _build():
    import oracle
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()
    yield
    _CACHE.clear()


def tickets(g, M):
    from fp8_block_scaled_router_gb300 import _lib as L
    v = L.moe_fp8_workspace_view(g.ws, g.shape)
    off = v.tickets - g.ws.data_ptr()
    n = min(g.shape.max_tokens, 16) * (g.H // 128)
    return g.ws[off: off + 4 * n].view(torch.int32)


# (workload, M): decode M=1 and M=2 (8 and 16 pairs), tiny (H=256: two K blocks, so most
# CTAs of a cluster route and compute nothing), the skewed verify router with its bias,
# wide h6144 (three K blocks per CTA), top-1 with 16 tokens; verify M=12 (96 pairs) is
# refused by the single launch
CASES = [("decode", 1), ("decode", 2), ("tiny", 4), ("verify_skewed", 1), ("wide", 1), ("wide", 4), ("top1", 16),
         ("verify", 12)]


@pytest.mark.parametrize("name,M", CASES, ids=[f"{n}-M{m}" for n, m in CASES])
def test_route_forward_matches_two_calls_and_oracle(name, M):
    from fp8_block_scaled_router_gb300 import _lib as L
    x = workload(name, M)
    g = GpuMoE(x, M)
    g.ws.fill_(0xFF)
    L.moe_fp8_workspace_init(g.ws, g.shape)
    hid = to_dev(x.hidden[:M])
    ids1 = torch.full((M, g.K), -7, dtype=torch.int32, device="cuda")
    w1 = torch.full((M, g.K), -7.0, dtype=torch.float32, device="cuda")
    out1 = torch.empty((M, g.H), dtype=torch.int16, device="cuda")
    rc = L.moe_fp8_route_forward_one_launch(hid, g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, out1, ids1,
                                            w1, g.ws, g.shape, check=False)
    # the single launch's limits: at most 16 routed pairs, at most 8 hidden B tiles per CTA
    supported = M * g.K <= 16 and (g.H // 128 + 15) // 16 * M <= 8
    if not supported:
        assert rc == 2  # MOE_ERR_UNSUPPORTED: only the two-call form takes it
        L.moe_fp8_route_forward(hid, g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, out1, ids1, w1, g.ws,
                                g.shape)
    else:
        assert rc == 0
    torch.cuda.synchronize()
    assert g.status() == 0
    ws = g.ws_arrays(M)
    # up to 64 routed pairs the intermediates are in pair order (the single launch or the two
    # pair kernels, both quantising the hidden row themselves)
    pair_order = M * g.K <= 64
    assert torch.all(tickets(g, M) == 0)
    ids_o, w_o = oracle_route(x, rows=slice(0, M))
    assert np.array_equal(ids1.cpu().numpy(), ids_o)
    assert np.all(np.abs(w1.cpu().numpy() - w_o) <= 2e-6 * w_o)
    out_o, dbg = oracle_forward(x, x.hidden[:M], ids_o, w_o, debug=True)
    if pair_order:  # the call's own intermediates: hidden codes, activation codes (pair order)
        assert np.array_equal(ws["qa"], dbg["qa"]) and np.array_equal(ws["sa"], dbg["sa"])
        ws["row_src"] = np.arange(M * g.K, dtype=np.int32)
        check_act(ws, dbg, g.K, f"route_forward {name} M={M}")
        check_out_given_act(u16(out1), out_o, ws, dbg, ids_o, w_o, x, f"route_forward {name} M={M}")
    # the two-call form on the same inputs: bitwise the same routing and output
    ids2 = torch.empty_like(ids1)
    w2 = torch.empty_like(w1)
    out2 = torch.empty_like(out1)
    L.moe_fp8_route_forward(hid, g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, out2, ids2, w2, g.ws, g.shape)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2) and torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert torch.equal(out1, out2)
    assert torch.all(tickets(g, M) == 0)


def test_route_forward_not_renormalised_and_rows_past_m():
    from fp8_block_scaled_router_gb300 import _lib as L
    x = workload("decode", 4)
    M = 1
    g = GpuMoE(x, 4)
    hid = to_dev(x.hidden[:M])
    ids = torch.full((4, g.K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((4, g.K), -7.0, dtype=torch.float32, device="cuda")
    out = torch.full((4, g.H), 0x7ABC, dtype=torch.int16, device="cuda")
    L.moe_fp8_route_forward_one_launch(hid, g.router, None, M, False, g.w13, g.s13, g.w2, g.s2, out, ids, w, g.ws,
                                       g.shape)
    torch.cuda.synchronize()
    ids_o, w_o = oracle_route(x, rows=slice(0, M), renorm=False)
    assert np.array_equal(ids[:M].cpu().numpy(), ids_o)
    assert np.all(np.abs(w[:M].cpu().numpy() - w_o) <= 2e-6 * w_o)
    assert torch.all(out[M:] == 0x7ABC) and torch.all(ids[M:] == -7) and torch.all(w[M:] == -7.0)
    ref = g.forward(hid, ids[:M].contiguous(), w[:M].contiguous(), M)
    torch.cuda.synchronize()
    assert torch.equal(out[:M], ref)


def test_route_forward_100_launches_and_graph_replay():
    """Bitwise identical over 100 eager launches and over CUDA-graph replays."""
    from fp8_block_scaled_router_gb300 import _lib as L
    x = workload("decode", 4)
    M = 1
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids = torch.empty((M, g.K), dtype=torch.int32, device="cuda")
    w = torch.empty((M, g.K), dtype=torch.float32, device="cuda")
    out = torch.empty((M, g.H), dtype=torch.int16, device="cuda")

    def call(st=None):
        L.moe_fp8_route_forward_one_launch(hid, g.router, g.bias, M, True, g.w13, g.s13, g.w2, g.s2, out, ids, w,
                                           g.ws, g.shape, stream=st)

    call()
    torch.cuda.synchronize()
    ref = (ids.clone(), w.clone(), out.clone())
    for it in range(100):
        out.zero_()
        call()
        assert torch.equal(out, ref[2]) and torch.equal(ids, ref[0]) and torch.equal(w, ref[1]), it
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for _ in range(4):
                call(s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(10):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref[2]) and torch.equal(ids, ref[0])
    assert g.status() == 0 and torch.all(tickets(g, M) == 0)
