"""CPU oracle for the routed FP8 block-scaled MoE FFN -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package. The product library never loads it and
shares no code with it: the oracle is a plain C++ restatement (``oracle.cpp``) built with
g++ and called through ctypes.

What it computes, step by step, is documented in ``oracle.cpp``; each function there names
the page and section it follows. Parity status: the codec, the quantiser, the router, the
RMSNorm in front of the layer and the block GEMMs are pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py``
against the E4M3 format definition, torch's float8 cast, float64 library matmuls with
rigorous error bounds, closed forms and brute force. The exact FP32 rounding order inside
the router's 128-wide chunks and the promotion chain is this library's contract reading
(the pages fix only that order is part of the contract); it is pinned at the value level,
not at the bit level.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_build/liboracle.so (g++, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared",
               "-fPIC", "-pthread", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Debug(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("qa", "sa", "g", "u", "gabs", "uabs", "act", "qact", "s2", "y")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.orc_e4m3_table.argtypes = [vp]
            lib.orc_e4m3_encode.argtypes = [vp, vp, i64]
            lib.orc_quantise.argtypes = [vp, i64, i32, vp, vp]
            lib.orc_bf16_round.argtypes = [vp, vp, i64]
            lib.orc_block_dot.argtypes = [vp, vp, i32]
            lib.orc_block_dot.restype = ctypes.c_float
            lib.orc_route.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
            lib.orc_route.restype = i32
            lib.orc_moe_forward.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                            vp, ctypes.POINTER(_Debug), i32]
            lib.orc_moe_forward.restype = i32
            lib.orc_down_combine.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32]
            lib.orc_down_combine.restype = i32
            lib.orc_rmsnorm.argtypes = [vp, vp, ctypes.c_float, i32, i32, vp, vp]
            lib.orc_rmsnorm.restype = i32
            lib.orc_e2m1_table.argtypes = [vp]
            lib.orc_ue8m0_decode.argtypes = [vp, vp, i64]
            lib.orc_mx_row.argtypes = [vp, vp, vp, vp, i32]
            lib.orc_mx_row.restype = ctypes.c_float
            lib.orc_mxfp4_forward.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                              ctypes.POINTER(_Debug), i32]
            lib.orc_mxfp4_forward.restype = i32
            lib.orc_mxfp4_down_combine.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32]
            lib.orc_mxfp4_down_combine.restype = i32
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e4m3_table() -> np.ndarray:
    out = np.empty(256, np.float32)
    _load().orc_e4m3_table(_p(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32)
    q = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode(_p(x), _p(q), x.size)
    return q


def quantise(x, group: int = 128):
    """Q over consecutive groups along the last axis: returns (codes uint8, scales f32)."""
    x = _c(x, np.float32)
    assert x.shape[-1] % group == 0
    q = np.empty(x.shape, np.uint8)
    s = np.empty(x.shape[:-1] + (x.shape[-1] // group,), np.float32)
    _load().orc_quantise(_p(x), x.size, group, _p(q), _p(s))
    return q, s


def bf16_round(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_round(_p(x), _p(out), x.size)
    return out


def block_dot(a, w) -> float:
    a, w = _c(a, np.uint8), _c(w, np.uint8)
    assert a.size == w.size
    return float(_load().orc_block_dot(_p(a), _p(w), a.size))


def route(hidden, router_w, bias, top_k: int, renormalize: bool = True, want_logits=False):
    """hidden uint16(BF16) [M][H], router_w uint16(BF16) [H][E], bias f32 [E] or None."""
    hidden, router_w = _c(hidden, np.uint16), _c(router_w, np.uint16)
    M, H = hidden.shape
    E = router_w.shape[1]
    assert router_w.shape[0] == H
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((M, top_k), np.int32)
    w = np.empty((M, top_k), np.float32)
    logits = np.empty((M, E), np.float32) if want_logits else None
    rc = _load().orc_route(_p(hidden), _p(router_w), _p(b), M, H, E, top_k, int(bool(renormalize)),
                           _p(ids), _p(w), _p(logits))
    if rc != 0:
        raise ValueError("oracle route: unsupported sizes")
    return (ids, w, logits) if want_logits else (ids, w)


def moe_forward(hidden, ids, weights, w13, s13, w2, s2w, debug: bool = False, nthreads: int = 1):
    """Returns out uint16(BF16) [M][H] (and a dict of intermediates when debug)."""
    hidden = _c(hidden, np.uint16)
    ids, weights = _c(ids, np.int32), _c(weights, np.float32)
    w13, s13, w2, s2w = _c(w13, np.uint8), _c(s13, np.float32), _c(w2, np.uint8), _c(s2w, np.float32)
    M, H = hidden.shape
    K = ids.shape[1]
    E, twoI, H2 = w13.shape
    I = twoI // 2
    assert H2 == H and w2.shape == (E, H, I) and ids.shape == weights.shape == (M, K)
    assert s13.shape == (E, twoI // 128, H // 128) and s2w.shape == (E, H // 128, I // 128)
    out = np.empty((M, H), np.uint16)
    dbg = None
    arrays = {}
    if debug:
        arrays = dict(qa=np.zeros((M, H), np.uint8), sa=np.zeros((M, H // 128), np.float32),
                      g=np.zeros((M, K, I), np.float32), u=np.zeros((M, K, I), np.float32),
                      gabs=np.zeros((M, K, I), np.float32), uabs=np.zeros((M, K, I), np.float32),
                      act=np.zeros((M, K, I), np.float32), qact=np.zeros((M, K, I), np.uint8),
                      s2=np.zeros((M, K, I // 128), np.float32), y=np.zeros((M, K, H), np.float32))
        dbg = _Debug(**{k: v.ctypes.data for k, v in arrays.items()})
    rc = _load().orc_moe_forward(_p(hidden), _p(ids), _p(weights), M, H, I, E, K, _p(w13), _p(s13),
                                 _p(w2), _p(s2w), _p(out),
                                 ctypes.byref(dbg) if dbg is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle forward: unsupported sizes")
    return (out, arrays) if debug else out


def down_combine(qact, s2, ids, weights, w2, s2w, nthreads: int = 1):
    """Steps 6-7 from given activation codes qact uint8 [M][K][I] and scales s2 f32
    [M][K][I/128]: the down projection of every routed pair and the slot-order combine.
    Returns out uint16(BF16) [M][H]."""
    qact, s2 = _c(qact, np.uint8), _c(s2, np.float32)
    ids, weights = _c(ids, np.int32), _c(weights, np.float32)
    w2, s2w = _c(w2, np.uint8), _c(s2w, np.float32)
    M, K, I = qact.shape
    E, H, I2 = w2.shape
    assert I2 == I and s2.shape == (M, K, I // 128) and ids.shape == weights.shape == (M, K)
    out = np.empty((M, H), np.uint16)
    rc = _load().orc_down_combine(_p(qact), _p(s2), _p(ids), _p(weights), M, H, I, E, K, _p(w2), _p(s2w), _p(out),
                                  int(nthreads))
    if rc != 0:
        raise ValueError("oracle down_combine: unsupported sizes")
    return out


def rmsnorm(x, gamma, eps: float, want_rstd: bool = False):
    """x uint16(BF16) [M][H], gamma uint16(BF16) [H] -> y uint16(BF16) [M][H] (and r f32 [M])."""
    x, gamma = _c(x, np.uint16), _c(gamma, np.uint16)
    M, H = x.shape
    assert gamma.shape == (H,)
    y = np.empty((M, H), np.uint16)
    r = np.empty(M, np.float32)
    rc = _load().orc_rmsnorm(_p(x), _p(gamma), float(eps), M, H, _p(y), _p(r))
    if rc != 0:
        raise ValueError("oracle rmsnorm: unsupported sizes")
    return (y, r) if want_rstd else y


# ---- MXFP4 weight variant ---------------------------------------------------------------
def e2m1_table() -> np.ndarray:
    out = np.empty(16, np.float32)
    _load().orc_e2m1_table(_p(out))
    return out


def ue8m0_decode(e) -> np.ndarray:
    e = _c(e, np.uint8)
    out = np.empty(e.shape, np.float32)
    _load().orc_ue8m0_decode(_p(e), _p(out), e.size)
    return out


def mx_row(a, sa, wq, ws) -> float:
    """One MXFP4 block-scaled row: a E4M3 codes [K], sa f32 [K/128], wq packed [K/2], ws [K/32]."""
    a, sa, wq, ws = _c(a, np.uint8), _c(sa, np.float32), _c(wq, np.uint8), _c(ws, np.uint8)
    assert a.size % 128 == 0 and wq.size * 2 == a.size and ws.size * 32 == a.size and sa.size * 128 == a.size
    return float(_load().orc_mx_row(_p(a), _p(sa), _p(wq), _p(ws), a.size // 128))


def mxfp4_forward(hidden, ids, weights, w13q, w13s, w2q, w2s, debug: bool = False, nthreads: int = 1):
    """The layer with MXFP4 expert weights (codes [E][N][K/2], UE8M0 scales [E][N][K/32])."""
    hidden = _c(hidden, np.uint16)
    ids, weights = _c(ids, np.int32), _c(weights, np.float32)
    w13q, w13s, w2q, w2s = _c(w13q, np.uint8), _c(w13s, np.uint8), _c(w2q, np.uint8), _c(w2s, np.uint8)
    M, H = hidden.shape
    K = ids.shape[1]
    E, twoI, Hh = w13q.shape
    I = twoI // 2
    assert Hh * 2 == H and w13s.shape == (E, twoI, H // 32)
    assert w2q.shape == (E, H, I // 2) and w2s.shape == (E, H, I // 32) and ids.shape == weights.shape == (M, K)
    out = np.empty((M, H), np.uint16)
    dbg = None
    arrays = {}
    if debug:
        arrays = dict(qa=np.zeros((M, H), np.uint8), sa=np.zeros((M, H // 128), np.float32),
                      g=np.zeros((M, K, I), np.float32), u=np.zeros((M, K, I), np.float32),
                      gabs=np.zeros((M, K, I), np.float32), uabs=np.zeros((M, K, I), np.float32),
                      act=np.zeros((M, K, I), np.float32), qact=np.zeros((M, K, I), np.uint8),
                      s2=np.zeros((M, K, I // 128), np.float32), y=np.zeros((M, K, H), np.float32))
        dbg = _Debug(**{k: v.ctypes.data for k, v in arrays.items()})
    rc = _load().orc_mxfp4_forward(_p(hidden), _p(ids), _p(weights), M, H, I, E, K, _p(w13q), _p(w13s), _p(w2q),
                                   _p(w2s), _p(out), ctypes.byref(dbg) if dbg is not None else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle mxfp4 forward: unsupported sizes")
    return (out, arrays) if debug else out


def mxfp4_down_combine(qact, s2, ids, weights, w2q, w2s, nthreads: int = 1):
    qact, s2 = _c(qact, np.uint8), _c(s2, np.float32)
    ids, weights = _c(ids, np.int32), _c(weights, np.float32)
    w2q, w2s = _c(w2q, np.uint8), _c(w2s, np.uint8)
    M, K, I = qact.shape
    E, H, I2 = w2q.shape
    assert I2 * 2 == I and w2s.shape == (E, H, I // 32)
    out = np.empty((M, H), np.uint16)
    rc = _load().orc_mxfp4_down_combine(_p(qact), _p(s2), _p(ids), _p(weights), M, H, I, E, K, _p(w2q), _p(w2s),
                                        _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle mxfp4 down_combine: unsupported sizes")
    return out
