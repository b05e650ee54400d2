"""The layer with MXFP4 expert weights on the GPU (moe_mxfp4_forward, moe_mxfp4_route_forward)
against the oracle's MXFP4 layer, on seeded inputs of the amd-kernels MXFP4 shape token
(h6144_i768_e128_top4; token count a runtime argument) and a tiny shape that splits two K
blocks over a cluster with a one-stage pipeline.

Tolerances are those of the FP8 layer (tests/gpu_harness.py): hidden codes and scales
bit-exact; activation codes bit-exact except next to a rounding boundary (window from the
oracle's error-scale reference, the sum of |P_s * 2^(e_s - 127) * sa| over the sub-blocks);
out within max(2e-2 * rms, one BF16 step) given the activation codes. Also: skipped pairs,
extreme UE8M0 exponents (e = 0, a subnormal factor), determinism, and route_forward equal to
route then forward bit for bit.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle
    from fp8_block_scaled_router_gb300 import _lib as L
    from gpu_harness import NTHREADS, GpuMoE, check_act, check_out_given_act, check_permutation, to_dev, u16

PAIR_ROWS = 64  # up to this many routed rows the layer runs one unit per pair

_CACHE = {}


def workload(name, E=None, tokens=None):
    key = (name, E, tokens)
    if key not in _CACHE:
        _CACHE[key] = inputs.make_mx(name, E=E, tokens=tokens)
    return _CACHE[key]


@pytest.fixture(scope="module", autouse=True)
def _build():
    from fp8_block_scaled_router_gb300 import build
    build.build()
    oracle.build()
    yield
    _CACHE.clear()


def run_mx(g, hid, ids, w, M):
    out = torch.empty((M, g.H), dtype=torch.int16, device="cuda")
    L.moe_mxfp4_forward(hid, ids, w, M, g.w13, g.s13, g.w2, g.s2, out, g.ws, g.shape)
    return out


def check_against_oracle(x, g, M, ids_o, w_o, out, what):
    out_o, dbg = oracle.mxfp4_forward(x.hidden[:M], ids_o, w_o, x.w13, x.s13, x.w2, x.s2, debug=True,
                                      nthreads=NTHREADS)
    ws = g.ws_arrays(M)
    assert np.array_equal(ws["qa"], dbg["qa"]) and np.array_equal(ws["sa"], dbg["sa"]), what
    if M * g.K <= PAIR_ROWS:  # pair kernels: activation rows in pair order
        ws["row_src"] = np.arange(M * g.K, dtype=np.int32)
    else:                     # expert-grouped kernels: rows in the sort's order
        check_permutation(ws, ids_o, x.shape.num_experts)
        ws["row_src"] = ws["row_src"][: int(ws["offsets"][-1])]  # the placed rows (valid ids)
    valid = (ids_o >= 0) & (ids_o < x.shape.num_experts)
    if valid.all():
        check_act(ws, dbg, g.K, what)
    check_out_given_act(u16(out), out_o, ws, dbg, ids_o, w_o, x, what,
                        down_combine=lambda q, s, i, w: oracle.mxfp4_down_combine(q, s, i, w, x.w2, x.s2,
                                                                                  nthreads=NTHREADS))


# pair kernels up to 64 routed rows, expert-grouped kernels above (groups of up to 16 rows of
# one expert; at M=256 over 16 experts each expert spans about four groups)
CASES = [("tiny_mxfp4", None, 1), ("tiny_mxfp4", None, 4), ("wide_mxfp4", 16, 1), ("wide_mxfp4", 16, 4),
         ("wide_mxfp4", 16, 16), ("wide_mxfp4", 16, 32), ("wide_mxfp4", 16, 64), ("wide_mxfp4", 16, 256),
         ("wide_mxfp4", None, 1), ("wide_mxfp4", None, 64)]


@pytest.mark.parametrize("name,E,M", CASES, ids=[f"{n}-E{e or 'full'}-M{m}" for n, e, m in CASES])
def test_mxfp4_forward_against_oracle(name, E, M):
    x = workload(name, E=E, tokens=max(64, M) if name == "wide_mxfp4" else None)
    g = GpuMoE(x, M)
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, None, x.shape.top_k)
    out = run_mx(g, to_dev(x.hidden[:M]), to_dev(ids_o), to_dev(w_o), M)
    torch.cuda.synchronize()
    assert g.status() == 0
    check_against_oracle(x, g, M, ids_o, w_o, out, f"{name} E={x.shape.num_experts} M={M}")


def test_mxfp4_skipped_pairs_flagged():
    x = workload("tiny_mxfp4")
    M = 4
    g = GpuMoE(x, M)
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, None, x.shape.top_k)
    bad = ids_o.copy()
    bad[0, 1] = -1
    bad[2, 0] = 99
    out = run_mx(g, to_dev(x.hidden[:M]), to_dev(bad), to_dev(w_o), M)
    torch.cuda.synchronize()
    assert g.status() & L.STATUS_BAD_EXPERT_ID
    check_against_oracle(x, g, M, bad, w_o, out, "tiny_mxfp4 skipped pairs")


def test_mxfp4_skipped_pairs_group_mode():
    """Skipped pairs with the expert-grouped kernels (48 tokens x top-2 = 96 routed rows)."""
    x = workload("tiny_mxfp4", tokens=48)
    M = 48
    g = GpuMoE(x, M)
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, None, x.shape.top_k)
    bad = ids_o.copy()
    bad[0, 1] = -1
    bad[7, 0] = 99
    bad[30, 1] = -3
    out = run_mx(g, to_dev(x.hidden[:M]), to_dev(bad), to_dev(w_o), M)
    torch.cuda.synchronize()
    assert g.status() & L.STATUS_BAD_EXPERT_ID  # the sort skips and flags them
    check_against_oracle(x, g, M, bad, w_o, out, "tiny_mxfp4 skipped pairs, group mode")


def test_mxfp4_extreme_exponents():
    """UE8M0 exponents 0 (2^-127, a subnormal factor), 1 and 127..160 mixed in every row: the
    GPU's FP32 products of P_s and the factor keep subnormals as the oracle's do."""
    x0 = workload("tiny_mxfp4")
    rng = np.random.default_rng(12345)
    s13 = x0.s13.copy()
    s2 = x0.s2.copy()
    for s in (s13, s2):
        pick = rng.random(s.shape)
        s[pick < 0.15] = 0
        s[(pick >= 0.15) & (pick < 0.25)] = 1
        big = (pick >= 0.25) & (pick < 0.35)
        s[big] = rng.integers(127, 161, size=int(big.sum()))
    import dataclasses
    x = dataclasses.replace(x0, s13=s13, s2=s2)
    M = 4
    g = GpuMoE(x, M)
    ids_o, w_o = oracle.route(x.hidden[:M], x.router_w, None, x.shape.top_k)
    out = run_mx(g, to_dev(x.hidden[:M]), to_dev(ids_o), to_dev(w_o), M)
    torch.cuda.synchronize()
    assert g.status() == 0
    check_against_oracle(x, g, M, ids_o, w_o, out, "tiny_mxfp4 extreme exponents")


def test_mxfp4_deterministic_route_forward_and_stages_equal():
    """Two runs bit-identical; moe_mxfp4_route_forward == moe_route + moe_mxfp4_forward ==
    moe_mxfp4_gate_up_direct + moe_mxfp4_down_combine, bit for bit."""
    x = workload("wide_mxfp4", E=16, tokens=64)
    M = 16
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    a = run_mx(g, hid, ids, w, M)
    b = run_mx(g, hid, ids, w, M)
    out = torch.empty_like(a)
    ids2 = torch.empty_like(ids)
    w2 = torch.empty_like(w)
    L.moe_mxfp4_route_forward(hid, g.router, None, M, True, g.w13, g.s13, g.w2, g.s2, out, ids2, w2, g.ws, g.shape)
    staged = torch.empty_like(a)
    L.moe_mxfp4_gate_up_direct(hid, ids, M, g.w13, g.s13, g.ws, g.shape)
    L.moe_mxfp4_down_combine(ids, w, M, g.w2, g.s2, staged, g.ws, g.shape)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(ids, ids2) and torch.equal(w, w2) and torch.equal(a, out)
    assert torch.equal(a, staged)
    assert g.status() == 0


def test_mxfp4_group_mode_stages_equal_forward():
    """Above 64 routed rows: moe_fp8_prepare + moe_mxfp4_gate_up + moe_mxfp4_down +
    moe_fp8_combine == moe_mxfp4_forward, bit for bit (48 tokens x top-4 = 192 rows)."""
    x = workload("wide_mxfp4", E=16, tokens=64)
    M = 48
    g = GpuMoE(x, M)
    hid = to_dev(x.hidden[:M])
    ids, w = g.route(hid, M)
    a = run_mx(g, hid, ids, w, M)
    staged = torch.empty_like(a)
    L.moe_fp8_prepare(hid, ids, M, g.ws, g.shape)
    L.moe_mxfp4_gate_up(g.w13, g.s13, M, g.ws, g.shape)
    L.moe_mxfp4_down(g.w2, g.s2, M, g.ws, g.shape)
    L.moe_fp8_combine(w, M, staged, g.ws, g.shape)
    torch.cuda.synchronize()
    assert torch.equal(a, staged)
    assert g.status() == 0
