"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library must load and export every function include/moe_fp8.h declares, and every
validation error path must return its status before any CUDA call (the netra-kernel
README's exact contract guards: an unsupported contract is refused, never approximated).
Each call below fails validation, so no kernel is ever launched with these fake pointers.
"""
import ctypes
import os
import re
import subprocess

import pytest

from fp8_block_scaled_router_gb300 import _lib as L
from fp8_block_scaled_router_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fp8.h")

FAKE = 0x10000  # 16-byte aligned, never dereferenced (validation fails first)
MIS = 0x10008   # misaligned


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(L.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for f in declared_functions():
        assert f in syms, f
        assert hasattr(lib, f)


def test_version(lib):
    assert "sm_103a" in L.moe_fp8_version()


def shape(**kw):
    d = dict(hidden=2048, inter=768, num_experts=128, top_k=8, max_tokens=16)
    d.update(kw)
    return L.make_shape(**d)


@pytest.mark.parametrize("kw", [dict(hidden=200), dict(hidden=0), dict(hidden=16384), dict(inter=100),
                                dict(inter=8192), dict(num_experts=100), dict(num_experts=512),
                                dict(top_k=0), dict(top_k=17), dict(num_experts=8, top_k=9),
                                dict(max_tokens=0)])
def test_unsupported_shapes(lib, kw):
    s = shape(**kw)
    assert L.moe_fp8_workspace_bytes(s) == 0
    code = L.moe_route(FAKE, FAKE, None, 1, s, 1, FAKE, FAKE, stream=0, check=False)
    assert code == 2  # MOE_ERR_UNSUPPORTED
    code = L.moe_fp8_forward(FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, s, stream=0,
                             ws_bytes=1 << 40, check=False)
    assert code == 2


def test_workspace_size_monotone_and_aligned(lib):
    a = L.moe_fp8_workspace_bytes(shape(max_tokens=1))
    b = L.moe_fp8_workspace_bytes(shape(max_tokens=64))
    c = L.moe_fp8_workspace_bytes(shape(max_tokens=4096))
    assert 0 < a < b < c and a % 256 == 0 and c % 256 == 0
    # the y buffer alone (R x H FP32) is part of it
    assert c >= 4096 * 8 * 2048 * 4


def test_forward_argument_errors(lib):
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    args = [FAKE] * 8
    # M out of range
    for M in (-1, 17):
        assert L.moe_fp8_forward(*args[:3], M, *args[3:8], FAKE, s, stream=0, ws_bytes=need,
                                 check=False) == 1
    # each null / misaligned pointer
    for i in range(8):
        for bad in (0, MIS):
            a = list(args)
            a[i] = bad
            assert L.moe_fp8_forward(*a[:3], 4, *a[3:8], FAKE, s, stream=0, ws_bytes=need,
                                     check=False) == 1, (i, bad)
    # workspace null, misaligned, too small
    assert L.moe_fp8_forward(*args[:3], 4, *args[3:8], 0, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_forward(*args[:3], 4, *args[3:8], MIS, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_forward(*args[:3], 4, *args[3:8], FAKE, s, stream=0, ws_bytes=need - 1,
                             check=False) == 3


def test_stage_and_route_argument_errors(lib):
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    assert L.moe_fp8_prepare(0, FAKE, 1, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_prepare(FAKE, FAKE, 1, FAKE, s, stream=0, ws_bytes=16, check=False) == 3
    assert L.moe_fp8_gate_up(FAKE, MIS, 1, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_down(FAKE, FAKE, 99, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_combine(FAKE, 1, 0, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_route(FAKE, FAKE, MIS, 1, s, 1, FAKE, FAKE, stream=0, check=False) == 1
    assert L.moe_route(FAKE, 0, None, 1, s, 1, FAKE, FAKE, stream=0, check=False) == 1
    assert L.moe_route(FAKE, FAKE, None, -3, s, 1, FAKE, FAKE, stream=0, check=False) == 1
    assert L.moe_fp8_workspace_init(FAKE, s, stream=0, ws_bytes=need - 256, check=False) == 3
    assert L.moe_fp8_read_status(0, FAKE, stream=0, check=False) == 1
    v = L.WsView()
    assert lib.moe_fp8_workspace_view(FAKE, 0, ctypes.byref(s), ctypes.byref(v)) == 3


def test_norm_argument_errors(lib):
    """The RMSNorm entry points refuse a null or misaligned weight and an eps that is not a
    finite positive number (eps = 0 would make an all-zero row 0 * inf = NaN)."""
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    calls = {
        "rmsnorm": lambda g, e, M=1: L.moe_rmsnorm(FAKE, g, e, M, FAKE, s, stream=0, check=False),
        "norm_route": lambda g, e, M=1: L.moe_norm_route(FAKE, g, e, FAKE, None, M, s, 1, FAKE, FAKE, stream=0,
                                                          check=False),
        "norm_forward": lambda g, e, M=1: L.moe_fp8_norm_forward(FAKE, g, e, FAKE, FAKE, M, FAKE, FAKE, FAKE, FAKE,
                                                                  FAKE, FAKE, s, stream=0, ws_bytes=need, check=False),
        "norm_route_forward": lambda g, e, M=1: L.moe_fp8_norm_route_forward(
            FAKE, g, e, FAKE, None, M, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, s, stream=0, ws_bytes=need,
            check=False),
    }
    for name, call in calls.items():
        for eps in (0.0, -1e-6, float("nan"), float("inf"), float("-inf")):
            assert call(FAKE, eps) == 1, (name, eps)
        assert call(0, 1e-6) == 1, name
        assert call(MIS, 1e-6) == 1, name
        assert call(FAKE, 1e-6, M=17) == 1, name   # above max_tokens
        assert call(FAKE, 1e-6, M=0) == 0, name    # no-op after validation
    assert L.moe_rmsnorm(MIS, FAKE, 1e-6, 1, FAKE, s, stream=0, check=False) == 1
    assert L.moe_rmsnorm(FAKE, FAKE, 1e-6, 1, 0, s, stream=0, check=False) == 1
    assert L.moe_rmsnorm(FAKE, FAKE, 1e-6, 1, FAKE, shape(hidden=200), stream=0, check=False) == 2
    assert L.moe_fp8_norm_forward(FAKE, FAKE, 1e-6, FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, s, stream=0,
                                  ws_bytes=need - 1, check=False) == 3


def test_verify_exact_batch_guard(lib):
    """The verify producer and reducer compile one profile (12 tokens, h2048 i768 e128 top-8):
    any other batch or shape is refused on the host before any launch."""
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)

    def produce(M, sh=s, nb=need, **bad):
        a = dict(hidden=FAKE, router_w=FAKE, bias=None, w13=FAKE, w13_scale=FAKE, w2=FAKE, w2_scale=FAKE,
                 topk_ids=FAKE, topk_w=FAKE)
        a.update(bad)
        return L.moe_fp8_verify_produce(a["hidden"], a["router_w"], a["bias"], M, 1, a["w13"], a["w13_scale"], a["w2"],
                                        a["w2_scale"], a["topk_ids"], a["topk_w"], FAKE, sh, stream=0, ws_bytes=nb,
                                        check=False)

    for M in (0, 1, 11, 13, 16):
        assert produce(M) == 2, M
        assert L.moe_fp8_verify_reduce(FAKE, M, FAKE, FAKE, s, stream=0, ws_bytes=need, check=False) == 2, M
    for kw in (dict(hidden=4096), dict(inter=1024), dict(num_experts=64), dict(top_k=4)):
        s2 = shape(**kw)
        n2 = L.moe_fp8_workspace_bytes(s2)
        assert produce(12, s2, n2) == 2, kw
        assert L.moe_fp8_verify_reduce(FAKE, 12, FAKE, FAKE, s2, stream=0, ws_bytes=n2, check=False) == 2, kw
    assert produce(12, shape(max_tokens=8), L.moe_fp8_workspace_bytes(shape(max_tokens=8))) == 1  # M > max_tokens
    for name in ("hidden", "router_w", "w13", "w13_scale", "w2", "w2_scale", "topk_ids", "topk_w"):
        assert produce(12, **{name: 0}) == 1, name
        assert produce(12, **{name: MIS}) == 1, name
    assert produce(12, bias=MIS) == 1
    assert produce(12, nb=need - 1) == 3
    assert L.moe_fp8_verify_reduce(0, 12, FAKE, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_fp8_verify_reduce(FAKE, 12, MIS, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    # the one-launch producer keeps the same guard
    for M in (0, 11, 13):
        assert L.moe_fp8_verify_produce_one_launch(FAKE, FAKE, None, M, 1, *[FAKE] * 6, FAKE, s, stream=0,
                                                   ws_bytes=need, check=False) == 2, M
    assert L.moe_fp8_verify_produce_one_launch(FAKE, FAKE, None, 12, 1, *[FAKE] * 6, FAKE, shape(top_k=4), stream=0,
                                               ws_bytes=L.moe_fp8_workspace_bytes(shape(top_k=4)), check=False) == 2
    assert L.moe_fp8_verify_produce_one_launch(MIS, FAKE, None, 12, 1, *[FAKE] * 6, FAKE, s, stream=0, ws_bytes=need,
                                               check=False) == 1


def test_partials_and_pair_reducer_argument_errors(lib):
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    args = [FAKE] * 7  # hidden, ids, w13, w13_scale, w2, w2_scale, y_out
    for i in range(7):
        for bad in (0, MIS):
            a = list(args)
            a[i] = bad
            assert L.moe_fp8_forward_partials(a[0], a[1], 4, a[2], a[3], a[4], a[5], a[6], FAKE, s, stream=0,
                                              ws_bytes=need, check=False) == 1, (i, bad)
    assert L.moe_fp8_forward_partials(*args[:2], 4, *args[2:], FAKE, s, stream=0, ws_bytes=need - 1, check=False) == 3
    assert L.moe_fp8_forward_partials(*args[:2], 0, *args[2:], FAKE, s, stream=0, ws_bytes=need, check=False) == 0
    assert L.moe_fp8_forward_partials(*args[:2], 17, *args[2:], FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    for i in range(4):
        a = [FAKE] * 4
        a[i] = MIS
        assert L.moe_fp8_combine_pairs(a[0], a[1], a[2], 4, a[3], s, stream=0, check=False) == 1, i
    assert L.moe_fp8_combine_pairs(FAKE, FAKE, FAKE, 0, FAKE, s, stream=0, check=False) == 0
    assert L.moe_fp8_combine_pairs(FAKE, FAKE, FAKE, 4, FAKE, shape(hidden=200), stream=0, check=False) == 2


def test_gate_up_prefetch_argument_errors(lib):
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    for i in range(6):  # hidden, ids, w13, w13_scale, w2, w2_scale
        for bad in (0, MIS):
            a = [FAKE] * 6
            a[i] = bad
            assert L.moe_fp8_gate_up_prefetch(a[0], a[1], 1, *a[2:], FAKE, s, stream=0, ws_bytes=need,
                                              check=False) == 1, (i, bad)
    assert L.moe_fp8_gate_up_prefetch(*[FAKE] * 2, 1, *[FAKE] * 4, FAKE, s, stream=0, ws_bytes=need - 1,
                                      check=False) == 3
    assert L.moe_fp8_gate_up_prefetch(*[FAKE] * 2, 0, *[FAKE] * 4, FAKE, s, stream=0, ws_bytes=need,
                                      check=False) == 0


def test_mxfp4_argument_errors(lib):
    """moe_mxfp4_forward / moe_mxfp4_route_forward and the two stage calls: null or misaligned
    pointers, a short workspace, M = 0; the stage calls (pair kernels) refuse more than 256
    routed rows."""
    s = shape(max_tokens=64)
    need = L.moe_fp8_workspace_bytes(s)
    for i in range(8):  # hidden, ids, w, w13q, w13_scale, w2q, w2_scale, out
        for bad in (0, MIS):
            a = [FAKE] * 8
            a[i] = bad
            assert L.moe_mxfp4_forward(a[0], a[1], a[2], 4, *a[3:], FAKE, s, stream=0, ws_bytes=need,
                                       check=False) == 1, (i, bad)
    f = [FAKE] * 8
    for i in (3, 5):  # the packed weight codes must be 32-byte aligned
        a = list(f)
        a[i] = FAKE + 16
        assert L.moe_mxfp4_forward(a[0], a[1], a[2], 4, *a[3:], FAKE, s, stream=0, ws_bytes=need,
                                   check=False) == 1, i
    assert L.moe_mxfp4_gate_up_direct(FAKE, FAKE, 4, FAKE + 16, FAKE, FAKE, s, stream=0, ws_bytes=need,
                                      check=False) == 1
    assert L.moe_mxfp4_down_combine(FAKE, FAKE, 4, FAKE + 16, FAKE, FAKE, FAKE, s, stream=0, ws_bytes=need,
                                    check=False) == 1
    assert L.moe_mxfp4_forward(*f[:3], 4, *f[3:], FAKE, s, stream=0, ws_bytes=need - 1, check=False) == 3
    assert L.moe_mxfp4_forward(*f[:3], 4, *f[3:], MIS, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_mxfp4_forward(*f[:3], 0, *f[3:], FAKE, s, stream=0, ws_bytes=need, check=False) == 0
    assert L.moe_mxfp4_forward(*f[:3], 4, *f[3:], FAKE, shape(hidden=200), stream=0, ws_bytes=need,
                               check=False) == 2
    r = [FAKE] * 11  # hidden, router, (bias), w13q, w13_scale, w2q, w2_scale, out, ids, w
    for i in [0, 1, 3, 4, 5, 6, 7, 8, 9]:
        a = list(r)
        a[i] = MIS
        assert L.moe_mxfp4_route_forward(a[0], a[1], None, 4, 1, a[3], a[4], a[5], a[6], a[7], a[8], a[9], FAKE,
                                         s, stream=0, ws_bytes=need, check=False) == 1, i
    assert L.moe_mxfp4_route_forward(FAKE, FAKE, MIS, 4, 1, *[FAKE] * 7, FAKE, s, stream=0, ws_bytes=need,
                                     check=False) == 1
    assert L.moe_mxfp4_route_forward(FAKE, FAKE, None, 0, 1, *[FAKE] * 7, FAKE, s, stream=0, ws_bytes=need,
                                     check=False) == 0
    for i in range(4):  # hidden, ids, w13q, w13_scale
        a = [FAKE] * 4
        a[i] = MIS
        assert L.moe_mxfp4_gate_up_direct(a[0], a[1], 4, a[2], a[3], FAKE, s, stream=0, ws_bytes=need,
                                          check=False) == 1, i
    assert L.moe_mxfp4_gate_up_direct(FAKE, FAKE, 33, FAKE, FAKE, FAKE, s, stream=0, ws_bytes=need, check=False) == 2
    for i in range(5):  # ids, w, w2q, w2_scale, out
        a = [FAKE] * 5
        a[i] = 0
        assert L.moe_mxfp4_down_combine(a[0], a[1], 4, a[2], a[3], a[4], FAKE, s, stream=0, ws_bytes=need,
                                        check=False) == 1, i
    assert L.moe_mxfp4_down_combine(*[FAKE] * 2, 4, *[FAKE] * 3, FAKE, s, stream=0, ws_bytes=need - 1,
                                    check=False) == 3
    # group-mode stage calls: alignment, a short workspace, too few rows to have been sorted
    assert L.moe_mxfp4_gate_up(FAKE + 16, FAKE, 16, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_mxfp4_down(FAKE, MIS, 16, FAKE, s, stream=0, ws_bytes=need, check=False) == 1
    assert L.moe_mxfp4_gate_up(FAKE, FAKE, 16, FAKE, s, stream=0, ws_bytes=need - 1, check=False) == 3
    assert L.moe_mxfp4_gate_up(FAKE, FAKE, 8, FAKE, s, stream=0, ws_bytes=need, check=False) == 2  # 64 rows
    assert L.moe_mxfp4_down(FAKE, FAKE, 8, FAKE, s, stream=0, ws_bytes=need, check=False) == 2
    assert L.moe_mxfp4_down(FAKE, FAKE, 0, FAKE, s, stream=0, ws_bytes=need, check=False) == 0


def test_zero_tokens_is_a_no_op(lib):
    """M = 0 returns MOE_OK after validation without touching the GPU (fake pointers)."""
    s = shape()
    need = L.moe_fp8_workspace_bytes(s)
    assert L.moe_route(FAKE, FAKE, None, 0, s, 1, FAKE, FAKE, stream=0, check=False) == 0
    assert L.moe_fp8_forward(FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, s, stream=0,
                             ws_bytes=need, check=False) == 0


def test_workspace_view_offsets(lib):
    s = shape(max_tokens=4)
    need = L.moe_fp8_workspace_bytes(s)
    v = L.moe_fp8_workspace_view(FAKE, s, ws_bytes=need)
    offs = [v.qa, v.sa, v.expert_offsets, v.row_src, v.perm_row, v.act, v.act_scale, v.y]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and offs[0] > FAKE and v.y < FAKE + need
    assert v.y + 4 * 8 * 2048 * 4 <= FAKE + need
