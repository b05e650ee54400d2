"""ctypes binding of libmoe_fp8.so (the C ABI of include/moe_fp8.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (or raw integer device pointers); the stream defaults to
torch's current stream. A non-zero status raises :class:`MoEError` unless ``check=False``.
The library must have been built (``fp8_block_scaled_router_gb300.build``); a missing
library raises at load time -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

_lock = threading.Lock()
_lib = None

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_LAUNCH"}
STATUS_BAD_EXPERT_ID = 0x1
STATUS_WAIT_TIMEOUT = 0x2

EXPORTS = ("moe_fp8_version", "moe_fp8_workspace_bytes", "moe_fp8_workspace_init", "moe_route",
           "moe_fp8_forward", "moe_fp8_prepare", "moe_fp8_gate_up", "moe_fp8_down",
           "moe_fp8_combine", "moe_fp8_workspace_view", "moe_fp8_read_status",
           "moe_fp8_forward_noalloc", "moe_fp8_gate_up_direct", "moe_fp8_down_combine",
           "moe_fp8_route_forward_host", "moe_fp8_route_forward_pinned", "moe_fp8_selftest_wait",
           "moe_fp8_route_forward", "moe_fp8_route_forward_one_launch", "moe_rmsnorm", "moe_norm_route",
           "moe_fp8_norm_forward", "moe_fp8_norm_route_forward", "moe_fp8_verify_produce",
           "moe_fp8_verify_reduce", "moe_fp8_forward_partials", "moe_fp8_combine_pairs", "moe_mxfp4_forward",
           "moe_mxfp4_route_forward", "moe_mxfp4_gate_up_direct", "moe_mxfp4_down_combine",
           "moe_mxfp4_gate_up", "moe_mxfp4_down", "moe_fp8_gate_up_prefetch",
           "moe_fp8_verify_produce_one_launch")


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32)]


class WsView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("qa", "sa", "row_src", "perm_row", "act", "act_scale", "y", "expert_offsets", "topk_ids",
                 "topk_w", "tickets")]


def load(path: str = LIB):
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libmoe_fp8.so not built ({path}); run "
                                   "python -m fp8_block_scaled_router_gb300.build")
            lib = ctypes.CDLL(path)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            sp = ctypes.POINTER(Shape)
            lib.moe_fp8_version.restype = ctypes.c_char_p
            lib.moe_fp8_workspace_bytes.argtypes = [sp]
            lib.moe_fp8_workspace_bytes.restype = sz
            lib.moe_fp8_workspace_init.argtypes = [vp, sz, sp, vp]
            lib.moe_route.argtypes = [vp, vp, vp, i32, sp, i32, vp, vp, vp]
            lib.moe_fp8_forward.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_prepare.argtypes = [vp, vp, i32, vp, sz, sp, vp]
            lib.moe_fp8_gate_up.argtypes = [vp, vp, i32, vp, sz, sp, vp]
            lib.moe_fp8_down.argtypes = [vp, vp, i32, vp, sz, sp, vp]
            lib.moe_fp8_combine.argtypes = [vp, i32, vp, vp, sz, sp, vp]
            lib.moe_fp8_workspace_view.argtypes = [vp, sz, sp, ctypes.POINTER(WsView)]
            lib.moe_fp8_read_status.argtypes = [vp, vp, vp]
            lib.moe_fp8_forward_noalloc.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, sp, vp]
            lib.moe_fp8_gate_up_direct.argtypes = [vp, vp, i32, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_down_combine.argtypes = [vp, vp, i32, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_route_forward_host.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_route_forward_pinned.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_selftest_wait.argtypes = [vp, sz, sp, ctypes.c_uint32, vp]
            lib.moe_fp8_route_forward.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_route_forward_one_launch.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                                             sp, vp]
            f32 = ctypes.c_float
            lib.moe_rmsnorm.argtypes = [vp, vp, f32, i32, vp, sp, vp]
            lib.moe_norm_route.argtypes = [vp, vp, f32, vp, vp, i32, sp, i32, vp, vp, vp]
            lib.moe_fp8_norm_forward.argtypes = [vp, vp, f32, vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_norm_route_forward.argtypes = [vp, vp, f32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                                       sz, sp, vp]
            lib.moe_fp8_verify_produce.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_verify_produce_one_launch.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                                              sp, vp]
            lib.moe_fp8_verify_reduce.argtypes = [vp, i32, vp, vp, sz, sp, vp]
            lib.moe_fp8_forward_partials.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_combine_pairs.argtypes = [vp, vp, vp, i32, vp, sp, vp]
            lib.moe_mxfp4_forward.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_fp8_gate_up_prefetch.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_mxfp4_gate_up.argtypes = [vp, vp, i32, vp, sz, sp, vp]
            lib.moe_mxfp4_down.argtypes = [vp, vp, i32, vp, sz, sp, vp]
            lib.moe_mxfp4_gate_up_direct.argtypes = [vp, vp, i32, vp, vp, vp, sz, sp, vp]
            lib.moe_mxfp4_down_combine.argtypes = [vp, vp, i32, vp, vp, vp, vp, sz, sp, vp]
            lib.moe_mxfp4_route_forward.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, sp, vp]
            for f in EXPORTS[2:]:
                if f != "moe_fp8_workspace_bytes":
                    getattr(lib, f).restype = i32
            _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _nbytes(x):
    return x if isinstance(x, int) else x.numel() * x.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code, check):
    if check and code != 0:
        raise MoEError(fn, code)
    return code


def make_shape(hidden, inter, num_experts, top_k, max_tokens) -> Shape:
    return Shape(hidden, inter, num_experts, top_k, max_tokens)


def moe_fp8_version() -> str:
    return load().moe_fp8_version().decode()


def moe_fp8_workspace_bytes(shape: Shape) -> int:
    return int(load().moe_fp8_workspace_bytes(ctypes.byref(shape)))


def moe_fp8_workspace_init(workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_workspace_init",
                  load().moe_fp8_workspace_init(_ptr(workspace), nb, ctypes.byref(shape), _stream(stream)),
                  check)


def moe_route(hidden, router_w, bias, M, shape: Shape, renormalize, topk_ids, topk_w, stream=None,
              check=True):
    return _check("moe_route", load().moe_route(_ptr(hidden), _ptr(router_w), _ptr(bias), int(M),
                                                ctypes.byref(shape), int(bool(renormalize)),
                                                _ptr(topk_ids), _ptr(topk_w), _stream(stream)), check)


def moe_fp8_forward(hidden, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out, workspace,
                    shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_forward", load().moe_fp8_forward(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w13), _ptr(w13_scale), _ptr(w2),
        _ptr(w2_scale), _ptr(out), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_forward(hidden, topk_ids, topk_w, M, w13q, w13_scale, w2q, w2_scale, out, workspace,
                      shape: Shape, stream=None, ws_bytes=None, check=True):
    """The layer with MXFP4 expert weights (packed E2M1 codes, UE8M0 scales per 32); see
    include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_forward", load().moe_mxfp4_forward(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w13q), _ptr(w13_scale), _ptr(w2q),
        _ptr(w2_scale), _ptr(out), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_gate_up_prefetch(hidden, topk_ids, M, w13, w13_scale, w2, w2_scale, workspace, shape: Shape,
                             stream=None, ws_bytes=None, check=True):
    """The forward's few-row gate/up launch (with the routed experts' w2 L2 prefetch)."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_gate_up_prefetch", load().moe_fp8_gate_up_prefetch(
        _ptr(hidden), _ptr(topk_ids), int(M), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale),
        _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_gate_up(w13q, w13_scale, M, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_gate_up", load().moe_mxfp4_gate_up(
        _ptr(w13q), _ptr(w13_scale), int(M), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_down(w2q, w2_scale, M, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_down", load().moe_mxfp4_down(
        _ptr(w2q), _ptr(w2_scale), int(M), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_gate_up_direct(hidden, topk_ids, M, w13q, w13_scale, workspace, shape: Shape, stream=None,
                             ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_gate_up_direct", load().moe_mxfp4_gate_up_direct(
        _ptr(hidden), _ptr(topk_ids), int(M), _ptr(w13q), _ptr(w13_scale), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_down_combine(topk_ids, topk_w, M, w2q, w2_scale, out, workspace, shape: Shape, stream=None,
                           ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_down_combine", load().moe_mxfp4_down_combine(
        _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w2q), _ptr(w2_scale), _ptr(out), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_mxfp4_route_forward(hidden, router_w, bias, M, renormalize, w13q, w13_scale, w2q, w2_scale, out, topk_ids,
                            topk_w, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """moe_route then moe_mxfp4_forward; see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_mxfp4_route_forward", load().moe_mxfp4_route_forward(
        _ptr(hidden), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)), _ptr(w13q), _ptr(w13_scale),
        _ptr(w2q), _ptr(w2_scale), _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_prepare(hidden, topk_ids, M, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_prepare", load().moe_fp8_prepare(
        _ptr(hidden), _ptr(topk_ids), int(M), _ptr(workspace), nb, ctypes.byref(shape),
        _stream(stream)), check)


def moe_fp8_gate_up(w13, w13_scale, M, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_gate_up", load().moe_fp8_gate_up(
        _ptr(w13), _ptr(w13_scale), int(M), _ptr(workspace), nb, ctypes.byref(shape),
        _stream(stream)), check)


def moe_fp8_down(w2, w2_scale, M, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_down", load().moe_fp8_down(
        _ptr(w2), _ptr(w2_scale), int(M), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)),
        check)


def moe_fp8_combine(topk_w, M, out, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_combine", load().moe_fp8_combine(
        _ptr(topk_w), int(M), _ptr(out), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)),
        check)


def moe_fp8_gate_up_direct(hidden, topk_ids, M, w13, w13_scale, workspace, shape: Shape, stream=None,
                           ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_gate_up_direct", load().moe_fp8_gate_up_direct(
        _ptr(hidden), _ptr(topk_ids), int(M), _ptr(w13), _ptr(w13_scale), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_down_combine(topk_ids, topk_w, M, w2, w2_scale, out, workspace, shape: Shape, stream=None,
                         ws_bytes=None, check=True):
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_down_combine", load().moe_fp8_down_combine(
        _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_workspace_view(workspace, shape: Shape, ws_bytes=None) -> WsView:
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    v = WsView()
    _check("moe_fp8_workspace_view",
           load().moe_fp8_workspace_view(_ptr(workspace), nb, ctypes.byref(shape), ctypes.byref(v)), True)
    return v


def moe_fp8_read_status(workspace, host_dst, stream=None, check=True):
    """host_dst: a pinned torch uint32/int32 CPU tensor of >= 1 element (or a host pointer)."""
    return _check("moe_fp8_read_status", load().moe_fp8_read_status(
        _ptr(workspace), _ptr(host_dst), _stream(stream)), check)


def moe_fp8_forward_noalloc(hidden, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out,
                            shape: Shape, stream=None, check=True):
    """moe_fp8_forward without a workspace (scratch compiled into the library; see
    include/moe_fp8.h for its limits and sharing rules)."""
    return _check("moe_fp8_forward_noalloc", load().moe_fp8_forward_noalloc(
        _ptr(hidden), _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w13), _ptr(w13_scale), _ptr(w2),
        _ptr(w2_scale), _ptr(out), ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_route_forward_host(host_hidden, host_out, M, router_w, bias, renormalize, w13, w13_scale, w2,
                               w2_scale, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """moe_route + moe_fp8_forward with hidden and out in (pinned) host memory; see
    include/moe_fp8.h. Returns at once; synchronise the stream before reading host_out."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_route_forward_host", load().moe_fp8_route_forward_host(
        _ptr(host_hidden), _ptr(host_out), int(M), _ptr(router_w), _ptr(bias), int(bool(renormalize)), _ptr(w13),
        _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_route_forward_pinned(host_hidden, host_out, M, router_w, bias, renormalize, w13, w13_scale, w2,
                                 w2_scale, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """moe_fp8_route_forward_host for page-locked host buffers (no pointer query); see
    include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_route_forward_pinned", load().moe_fp8_route_forward_pinned(
        _ptr(host_hidden), _ptr(host_out), int(M), _ptr(router_w), _ptr(bias), int(bool(renormalize)), _ptr(w13),
        _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_selftest_wait(workspace, shape: Shape, limit_us, stream=None, ws_bytes=None, check=True):
    """Bounded-wait self-check: sets MOE_STATUS_WAIT_TIMEOUT in the workspace status."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_selftest_wait", load().moe_fp8_selftest_wait(
        _ptr(workspace), nb, ctypes.byref(shape), int(limit_us), _stream(stream)), check)


def moe_fp8_route_forward(hidden, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale, out, topk_ids,
                          topk_w, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """Routing + the expert FFN in one call; see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_route_forward", load().moe_fp8_route_forward(
        _ptr(hidden), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)), _ptr(w13), _ptr(w13_scale),
        _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_route_forward_one_launch(hidden, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale, out,
                                     topk_ids, topk_w, workspace, shape: Shape, stream=None, ws_bytes=None,
                                     check=True):
    """Routing + the expert FFN as a single kernel launch (few routed pairs); see
    include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_route_forward_one_launch", load().moe_fp8_route_forward_one_launch(
        _ptr(hidden), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)), _ptr(w13), _ptr(w13_scale),
        _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), nb,
        ctypes.byref(shape), _stream(stream)), check)


def moe_rmsnorm(hidden, norm_weight, eps, M, out, shape: Shape, stream=None, check=True):
    """out = RMSNorm(hidden) (BF16 rows); see include/moe_fp8.h for the exact arithmetic."""
    return _check("moe_rmsnorm", load().moe_rmsnorm(
        _ptr(hidden), _ptr(norm_weight), float(eps), int(M), _ptr(out), ctypes.byref(shape), _stream(stream)), check)


def moe_norm_route(hidden, norm_weight, eps, router_w, bias, M, shape: Shape, renormalize, topk_ids, topk_w,
                   stream=None, check=True):
    """moe_route of the RMSNorm'd hidden (the router normalises as it reads)."""
    return _check("moe_norm_route", load().moe_norm_route(
        _ptr(hidden), _ptr(norm_weight), float(eps), _ptr(router_w), _ptr(bias), int(M), ctypes.byref(shape),
        int(bool(renormalize)), _ptr(topk_ids), _ptr(topk_w), _stream(stream)), check)


def moe_fp8_norm_forward(hidden, norm_weight, eps, topk_ids, topk_w, M, w13, w13_scale, w2, w2_scale, out,
                         workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """moe_fp8_forward of the RMSNorm'd hidden (the quantisers normalise as they read)."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_norm_forward", load().moe_fp8_norm_forward(
        _ptr(hidden), _ptr(norm_weight), float(eps), _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(w13),
        _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(workspace), nb, ctypes.byref(shape),
        _stream(stream)), check)


def moe_fp8_norm_route_forward(hidden, norm_weight, eps, router_w, bias, M, renormalize, w13, w13_scale, w2,
                               w2_scale, out, topk_ids, topk_w, workspace, shape: Shape, stream=None, ws_bytes=None,
                               check=True):
    """moe_fp8_route_forward of the RMSNorm'd hidden; see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_norm_route_forward", load().moe_fp8_norm_route_forward(
        _ptr(hidden), _ptr(norm_weight), float(eps), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)),
        _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(out), _ptr(topk_ids), _ptr(topk_w),
        _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_verify_produce(hidden, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale, topk_ids, topk_w,
                           workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """The verify_m12 producer (routing, gate/up, SiLU+quant, down partials); see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_verify_produce", load().moe_fp8_verify_produce(
        _ptr(hidden), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)), _ptr(w13), _ptr(w13_scale),
        _ptr(w2), _ptr(w2_scale), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), nb, ctypes.byref(shape),
        _stream(stream)), check)


def moe_fp8_verify_produce_one_launch(hidden, router_w, bias, M, renormalize, w13, w13_scale, w2, w2_scale,
                                      topk_ids, topk_w, workspace, shape: Shape, stream=None, ws_bytes=None,
                                      check=True):
    """The verify_m12 producer as one launch (opt-in); see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_verify_produce_one_launch", load().moe_fp8_verify_produce_one_launch(
        _ptr(hidden), _ptr(router_w), _ptr(bias), int(M), int(bool(renormalize)), _ptr(w13), _ptr(w13_scale),
        _ptr(w2), _ptr(w2_scale), _ptr(topk_ids), _ptr(topk_w), _ptr(workspace), nb, ctypes.byref(shape),
        _stream(stream)), check)


def moe_fp8_verify_reduce(topk_w, M, out, workspace, shape: Shape, stream=None, ws_bytes=None, check=True):
    """The verify_m12 route reducer (slot-order combine of the producer's partials)."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_verify_reduce", load().moe_fp8_verify_reduce(
        _ptr(topk_w), int(M), _ptr(out), _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_forward_partials(hidden, topk_ids, M, w13, w13_scale, w2, w2_scale, y_out, workspace, shape: Shape,
                             stream=None, ws_bytes=None, check=True):
    """Every routed pair's FP32 down projection in pair order (y_out [M*K][H]); see include/moe_fp8.h."""
    nb = _nbytes(workspace) if ws_bytes is None else ws_bytes
    return _check("moe_fp8_forward_partials", load().moe_fp8_forward_partials(
        _ptr(hidden), _ptr(topk_ids), int(M), _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(y_out),
        _ptr(workspace), nb, ctypes.byref(shape), _stream(stream)), check)


def moe_fp8_combine_pairs(y, topk_ids, topk_w, M, out, shape: Shape, stream=None, check=True):
    """The slot-order route reducer over pair-order FP32 rows y [M*K][H] -> out BF16 [M][H]."""
    return _check("moe_fp8_combine_pairs", load().moe_fp8_combine_pairs(
        _ptr(y), _ptr(topk_ids), _ptr(topk_w), int(M), _ptr(out), ctypes.byref(shape), _stream(stream)), check)
