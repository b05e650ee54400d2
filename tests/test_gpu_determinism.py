"""Determinism and graph replay (GPU).

docs/compiler/architecture.md reports repeated-launch determinism and exact graph replays
as acceptance evidence, and the amd-kernels README's reduction rule (fixed order, no
atomics) is what makes results reproducible: 100 launches must be bitwise identical.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import GpuMoE, to_dev


@pytest.fixture(scope="module", autouse=True)
def _build_lib():
    from fp8_block_scaled_router_gb300 import build
    build.build()


def _workload(name, M):
    if name == "grouped":  # 64 tokens x top-8 over 16 experts: the sorted-tile path
        return inputs.make("decode", E=16, tokens=M)
    if name == "groups":   # 32 tokens x top-8 over 16 experts: the expert-grouped pair kernels
        return inputs.make("decode", E=16, tokens=M)
    if name == "decode":
        return inputs.make(name, tokens=M)
    return inputs.make(name, M=M)


DET_CASES = [("decode", 1), ("verify", 12), ("tiny", 4), ("groups", 32), ("grouped", 64), ("wide", 1), ("wide", 64),
             ("prefill", 4096), ("prefill_zipf", 4096)]


@pytest.mark.parametrize("name,M", DET_CASES, ids=[f"{n}-M{m}" for n, m in DET_CASES])
def test_100_launches_bitwise_identical(name, M):
    """Route + forward 100 times on the same inputs: ids, weights, the activation codes and
    scales and the output are bitwise identical every time (compared on the device)."""
    from fp8_block_scaled_router_gb300 import _lib as L
    x = _workload(name, M)
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    given = None if x.ids is None else (to_dev(x.ids[:M]), to_dev(x.weights[:M]))
    v = L.moe_fp8_workspace_view(g.ws, g.shape)
    base = g.ws.data_ptr()
    R = M * g.K
    act = g.ws[v.act - base: v.act - base + R * g.I]
    act_s = g.ws[v.act_scale - base: v.act_scale - base + R * (g.I // 128) * 4]
    ref = None
    for it in range(100):
        ids, w = g.route(hid, M)
        fi, fw = given if given is not None else (ids, w)
        out = g.forward(hid, fi, fw, M)
        cur = (ids.clone(), w.view(torch.int32).clone(), out.clone(), act.clone(), act_s.clone())
        if ref is None:
            ref = cur
        else:
            for k, (a, b) in enumerate(zip(ref, cur)):
                assert torch.equal(a, b), f"launch {it} differs (output {k})"
    assert g.status() == 0


def test_graph_capture_replay_matches_eager():
    x = inputs.make("verify")
    M = 12
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    out_eager = g.forward(hid, ids, w, M).clone()
    ids_eager, w_eager = ids.clone(), w.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = torch.empty_like(out_eager)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            ids2, w2 = g.route(hid, M)
            g.forward(hid, ids2, w2, M, out=out)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(20):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_eager)
        assert torch.equal(ids2, ids_eager) and torch.equal(w2, w_eager)


@pytest.mark.parametrize("name,M", [("decode", 1), ("verify_skewed", 12), ("tiny", 4), ("groups", 32), ("grouped", 64)])
def test_forward_equals_stage_calls(name, M):
    """moe_fp8_forward (which may fuse stages) and the four stage calls give bitwise equal
    outputs: the fused kernels use the same arithmetic in the same order."""
    from fp8_block_scaled_router_gb300 import _lib as L
    x = _workload(name, M)
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    out_fused = g.forward(hid, ids, w, M).clone()
    out_staged = torch.empty_like(out_fused)
    L.moe_fp8_prepare(hid, ids, M, g.ws, g.shape)
    L.moe_fp8_gate_up(g.w13, g.s13, M, g.ws, g.shape)
    L.moe_fp8_down(g.w2, g.s2, M, g.ws, g.shape)
    L.moe_fp8_combine(w, M, out_staged, g.ws, g.shape)
    torch.cuda.synchronize()
    assert torch.equal(out_fused, out_staged)


def test_gate_up_prefetch_equals_direct():
    """The forward's few-row gate/up launch (with the w2 L2 prefetch) writes the same
    activation codes and scales as moe_fp8_gate_up_direct, bit for bit."""
    from fp8_block_scaled_router_gb300 import _lib as L
    x = _workload("decode", 4)
    g = GpuMoE(x, 4)
    hid = to_dev(x.hidden[:4])
    ids, w = g.route(hid, 4)
    L.moe_fp8_gate_up_direct(hid, ids, 4, g.w13, g.s13, g.ws, g.shape)
    a = g.ws_arrays(4)
    L.moe_fp8_gate_up_prefetch(hid, ids, 4, g.w13, g.s13, g.w2, g.s2, g.ws, g.shape)
    b = g.ws_arrays(4)
    torch.cuda.synchronize()
    assert np.array_equal(a["act"], b["act"]) and np.array_equal(a["act_scale"], b["act_scale"])
    assert np.array_equal(a["qa"], b["qa"]) and np.array_equal(a["sa"], b["sa"])
    assert g.status() == 0
