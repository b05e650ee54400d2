"""GPU parity: the CUDA library (called through its C ABI) against the CPU oracle on the same
seeded inputs, at every workload shape; tolerances are stated in tests/gpu_harness.py.

Workloads follow the netra-kernel pages' regimes for the Qwen3.6 FP8 MoE (decode M=1,
speculative verify M=12, prefill) and the amd-kernels wide-expert shape token
(h6144_i768_e128_top4, token count a runtime argument, CUDA-graph padding rows).
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import (GpuMoE, check_act, check_out, check_out_given_act, check_permutation,
                             oracle_forward, oracle_route, to_dev, u16)

_CACHE = {}


def workload(name, **kw):
    key = (name, tuple(sorted(kw.items())))
    if key not in _CACHE:
        _CACHE[key] = inputs.make(name, **kw)
    return _CACHE[key]


@pytest.fixture(scope="module", autouse=True)
def _build_lib():
    from fp8_block_scaled_router_gb300 import build
    import oracle
    build.build()
    oracle.build()
    yield
    _CACHE.clear()


def gpu_for(x, max_tokens):
    return GpuMoE(x, max_tokens)


# ------------------------------------------------------------------ routing
ROUTE_CASES = [("tiny", 4), ("decode", 64), ("decode", 1), ("verify", 12), ("verify_skewed", 12),
               ("wide", 64), ("prefill", 4096)]


@pytest.mark.parametrize("name,M", ROUTE_CASES, ids=[f"{n}-M{m}" for n, m in ROUTE_CASES])
def test_route_parity(name, M):
    x = workload(name) if name != "decode" else workload(name, tokens=64)
    g = gpu_for(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    torch.cuda.synchronize()
    ids_o, w_o = oracle_route(x, rows=slice(0, M))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    wg = w.cpu().numpy()
    assert np.all(np.abs(wg - w_o) <= 2e-6 * w_o)


# the many-token router (M >= 512, E in {32, 64, 128}): ragged last block, every expert
# count it covers, the bias of the skewed workload, both softmax domains
BIG_ROUTE = [("prefill", 128, 1000, True), ("prefill", 64, 512, True), ("prefill", 32, 777, False),
             ("verify_skewed", 128, 600, True), ("decode", 128, 544, False)]


@pytest.mark.parametrize("name,E,M,renorm", BIG_ROUTE, ids=[f"{n}-E{e}-M{m}-{r}" for n, e, m, r in BIG_ROUTE])
def test_route_many_tokens(name, E, M, renorm):
    x = workload(name, E=E, tokens=M) if name == "decode" else workload(name, E=E, M=M)
    g = gpu_for(x, M)
    ids, w = g.route(to_dev(x.hidden[:M]), M, renorm=renorm)
    torch.cuda.synchronize()
    ids_o, w_o = oracle_route(x, rows=slice(0, M), renorm=renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)


def test_route_many_tokens_ties():
    # zero hidden rows: every logit is +0, so the top-k are experts 0..K-1 with equal weights
    M = 640
    x = inputs.make("prefill", M=M, zero_rows=np.arange(0, M, 7))
    g = gpu_for(x, M)
    ids, w = g.route(to_dev(x.hidden[:M]), M)
    torch.cuda.synchronize()
    ids_o, w_o = oracle_route(x, rows=slice(0, M))
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.array_equal(ids_o[0], np.arange(x.shape.top_k))
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)


def test_route_not_renormalised():
    x = workload("decode", tokens=64)
    g = gpu_for(x, 64)
    ids, w = g.route(to_dev(x.hidden[:64]), 64, renorm=False)
    torch.cuda.synchronize()
    ids_o, w_o = oracle_route(x, rows=slice(0, 64), renorm=False)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.all(np.abs(w.cpu().numpy() - w_o) <= 2e-6 * w_o)


def test_route_rows_beyond_m_untouched():
    x = workload("verify")
    g = gpu_for(x, 12)
    ids = torch.full((16, 8), -777, dtype=torch.int32, device="cuda")
    w = torch.full((16, 8), -7.0, dtype=torch.float32, device="cuda")
    from fp8_block_scaled_router_gb300 import _lib as L
    L.moe_route(to_dev(x.hidden[:12]), g.router, g.bias, 12, g.shape, True, ids, w)
    torch.cuda.synchronize()
    assert torch.all(ids[12:] == -777) and torch.all(w[12:] == -7.0)


# ------------------------------------------------------------------ forward
def poison_workspace(g):
    """Stale contents must not matter: every value a test reads must be written by the call."""
    g.ws.fill_(0xFF)
    from fp8_block_scaled_router_gb300 import _lib as L
    L.moe_fp8_workspace_init(g.ws, g.shape)


def run_forward_case(x, M, max_tokens=None, zero_rows=None):
    g = gpu_for(x, max_tokens or M)
    poison_workspace(g)
    hidden = x.hidden[:M].copy()
    if zero_rows is not None:
        hidden[zero_rows] = 0
    if x.ids is not None:
        ids_o, w_o = x.ids[:M], x.weights[:M]
    else:
        import oracle
        ids_o, w_o = oracle.route(hidden, x.router_w, x.bias, x.shape.top_k)
    hid_d, ids_d = to_dev(hidden), to_dev(ids_o)
    out = g.forward(hid_d, ids_d, to_dev(w_o), M)
    torch.cuda.synchronize()
    # the hidden codes and scales as the forward's own quantiser wrote them (the few-row
    # gate/up kernel quantises in its prologue; the sorted path in its count+quantise pass)
    ws = g.ws_arrays(M)
    qa, sa = ws["qa"].copy(), ws["sa"].copy()
    # the few-row forward writes no permutation; the prepare stage fills those views (it
    # does not touch the activation codes)
    from fp8_block_scaled_router_gb300 import _lib as L
    L.moe_fp8_prepare(hid_d, ids_d, M, g.ws, g.shape)
    torch.cuda.synchronize()
    ws = g.ws_arrays(M)
    ws["qa"], ws["sa"] = qa, sa
    out_o, dbg = oracle_forward(x, hidden, ids_o, w_o, debug=True)
    dbg["w"] = w_o
    return g, ids_o, ws, u16(out), out_o, dbg


def check_all(x, M, ids_o, ws, out, out_o, dbg, what):
    assert np.array_equal(ws["qa"], dbg["qa"]), f"{what}: hidden codes"
    assert np.array_equal(ws["sa"], dbg["sa"]), f"{what}: hidden scales"
    check_permutation(ws, ids_o, x.shape.num_experts)
    check_act(ws, dbg, x.shape.top_k, what)
    check_out_given_act(out, out_o, ws, dbg, ids_o, dbg["w"], x, what)


FWD_CASES = [("tiny", 4), ("verify", 12), ("verify_skewed", 12)]


@pytest.mark.parametrize("name,M", FWD_CASES, ids=[f"{n}-M{m}" for n, m in FWD_CASES])
def test_forward_parity(name, M):
    x = workload(name)
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, M)
    check_all(x, M, ids_o, ws, out, out_o, dbg, name)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_wide_sweep_with_padding_rows(M):
    x = workload("wide")
    pad = inputs.wide_padding_rows(M)
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, M, max_tokens=64, zero_rows=pad)
    check_all(x, M, ids_o, ws, out, out_o, dbg, f"wide M={M}")
    if len(pad):
        assert np.all(out[pad] == 0)


def test_decode_tokens_one_per_launch():
    """Decode: one token per launch over 48 seeded tokens, each compared with the oracle."""
    x = workload("decode", tokens=48)
    g = gpu_for(x, 1)
    import oracle
    ids_o, w_o = oracle.route(x.hidden, x.router_w, None, 8)
    outs = []
    for t in range(48):
        outs.append(u16(g.forward(to_dev(x.hidden[t:t + 1]), to_dev(ids_o[t:t + 1]),
                                  to_dev(w_o[t:t + 1]), 1)))
    out_o = oracle_forward(x, x.hidden, ids_o, w_o)
    for t in range(48):
        check_out(outs[t], out_o[t:t + 1], f"decode token {t}")


def test_many_tiles_with_ragged_tails():
    """300 tokens over 16 experts (top-8): ~150 rows per expert, so experts span two
    128-row tiles with a ragged last tile; full oracle comparison."""
    x = workload("decode", E=16, tokens=300)
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, 300)
    counts = np.bincount(ids_o.ravel(), minlength=16)
    assert np.any(counts % 128 != 0) and counts.max() > 128
    check_all(x, 300, ids_o, ws, out, out_o, dbg, "ragged")


def test_expert_groups_spanning_several_groups():
    """The expert-grouped pair kernels (64 < routed rows <= 256) with experts holding more
    than one group of 16 rows: 32 tokens top-8 over 16 experts (256 rows, 16 per expert on
    average)."""
    x = workload("decode", E=16, tokens=32)
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, 32)
    counts = np.bincount(ids_o.ravel(), minlength=16)
    assert counts.max() > 16
    check_all(x, 32, ids_o, ws, out, out_o, dbg, "expert groups")


@pytest.mark.parametrize("name", ["prefill", "prefill_zipf"])
def test_prefill_full_size(name):
    """The full M=4096 launch against the oracle on every token: hidden codes and scales,
    the permutation, all 32768 routed rows' activation codes and scales, and the output."""
    x = workload(name)
    M = 4096
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, M)
    check_all(x, M, ids_o, ws, out, out_o, dbg, name)


def test_large_gate_values_sorted_tiles():
    """Gate/up values of tens (w13 block scales x 16, a power of two, so the codes are
    unchanged): the sorted-tile epilogue's SiLU must hold the activation-code window where
    exp(-g) is far from 1 in either direction. 300 tokens over 16 experts (sorted tiles)."""
    import dataclasses
    x = workload("decode", E=16, tokens=300)
    x = dataclasses.replace(x, s13=(x.s13 * np.float32(16.0)).astype(np.float32))
    _, ids_o, ws, out, out_o, dbg = run_forward_case(x, 300)
    assert np.abs(dbg["g"]).max() > 20 and dbg["g"].min() < -20
    check_all(x, 300, ids_o, ws, out, out_o, dbg, "large g (sorted)")


PAIR_DIRECT = [("verify_skewed", 12), ("decode", 32)]  # 96 and 256 routed rows


@pytest.mark.parametrize("name,M", PAIR_DIRECT, ids=[f"{n}-R{m * 8}" for n, m in PAIR_DIRECT])
def test_pair_kernels_against_oracle(name, M):
    """The two few-row kernels as direct calls (one unit per routed pair) above the 64 rows
    at which moe_fp8_forward switches to sorted tiles: hidden codes from the gate/up kernel's
    own quantiser, activation codes and scales in pair order, and the output."""
    from fp8_block_scaled_router_gb300 import _lib as L
    x = workload(name) if name != "decode" else workload(name, tokens=M)
    g = gpu_for(x, M)
    poison_workspace(g)
    import oracle
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, x.bias, x.shape.top_k)
    hid, ids, w = to_dev(x.hidden[:M]), to_dev(ids_o), to_dev(w_o)
    out = torch.empty((M, g.H), dtype=torch.int16, device="cuda")
    L.moe_fp8_gate_up_direct(hid, ids, M, g.w13, g.s13, g.ws, g.shape)
    L.moe_fp8_down_combine(ids, w, M, g.w2, g.s2, out, g.ws, g.shape)
    torch.cuda.synchronize()
    assert g.status() == 0
    ws = g.ws_arrays(M)
    out_o, dbg = oracle_forward(x, x.hidden[:M], ids_o, w_o, debug=True)
    assert np.array_equal(ws["qa"], dbg["qa"]) and np.array_equal(ws["sa"], dbg["sa"])
    ws["row_src"] = np.arange(M * g.K, dtype=np.int32)  # pair order
    check_act(ws, dbg, g.K, f"{name} direct R={M * g.K}")
    check_out_given_act(u16(out), out_o, ws, dbg, ids_o, w_o, x, f"{name} direct")


def test_output_rows_beyond_m_untouched():
    x = workload("verify")
    g = gpu_for(x, 16)
    import oracle
    ids_o, w_o = oracle.route(x.hidden[:12], x.router_w, None, 8)
    out = torch.full((16, 2048), 0x7ABC, dtype=torch.int16, device="cuda")
    g.forward(to_dev(x.hidden[:12]), to_dev(ids_o), to_dev(w_o), 12, out=out)
    torch.cuda.synchronize()
    assert torch.all(out[12:] == 0x7ABC)


def test_invalid_ids_flagged_and_skipped():
    x = workload("tiny")
    g = gpu_for(x, 4)
    import oracle
    ids_o, w_o = oracle.route(x.hidden, x.router_w, None, 2)
    bad = ids_o.copy()
    bad[0, 1] = -1
    bad[2, 0] = 99
    assert g.status() == 0
    out = u16(g.forward(to_dev(x.hidden), to_dev(bad), to_dev(w_o), 4))
    assert g.status() & 0x1
    out_o = oracle_forward(x, x.hidden, bad, w_o)
    check_out(out, out_o, "invalid ids")
    g2 = gpu_for(x, 4)
    g2.forward(to_dev(x.hidden), to_dev(ids_o), to_dev(w_o), 4)
    assert g2.status() == 0


def test_invalid_ids_grouped_path():
    # 48 tokens x 8 slots = 384 routed rows: expert-sorted tiles; invalid pairs are never
    # placed, so fewer rows than M*K are gathered and the GEMM tiles cover only valid rows
    M = 48
    x = workload("decode", tokens=M)
    g = gpu_for(x, M)
    g.ws.fill_(0xFF)  # stale workspace contents must not matter
    from fp8_block_scaled_router_gb300 import _lib as L
    L.moe_fp8_workspace_init(g.ws, g.shape)
    import oracle
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, None, 8)
    bad = ids_o.copy()
    bad[0, 1] = -1
    bad[5, 0] = 128
    bad[47, 7] = -5
    out = u16(g.forward(to_dev(x.hidden[:M]), to_dev(bad), to_dev(w_o), M))
    assert g.status() & 0x1
    check_out(out, oracle_forward(x, x.hidden[:M], bad, w_o), "invalid ids (grouped)")


def test_end_to_end_gpu_route_feeds_forward():
    x = workload("verify_skewed")
    g = gpu_for(x, 12)
    hid = to_dev(x.hidden[:12])
    ids, w = g.route(hid, 12)
    out = u16(g.forward(hid, ids, w, 12))
    import oracle
    ids_o, w_o = oracle.route(x.hidden[:12], x.router_w, x.bias, 8)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    check_out(out, oracle_forward(x, x.hidden[:12], ids_o, w_o), "e2e")
