"""Helpers for the GPU tests: run the library through its C ABI on seeded inputs and
compare with the oracle.

Tolerances (written out where they are checked):
* top-k ids, hidden FP8 codes and hidden scales: bit-exact;
* router weights: |w - w_oracle| <= 2e-6 * w_oracle;
* activation FP8 codes: bit-exact, except a code whose oracle pre-quantisation value v
  lies within ``window(v)`` of a rounding boundary (then one code step either way), where
  window(v) = 1e-6*|v| + 5e-6 * noise(v): 1e-6 relative, plus the first-order bound of the
  GPU's FP32 block sums (at most 64+16+1 roundings of terms whose magnitudes sum to the
  oracle's gabs/uabs, 81 * 2^-24 < 5e-6) propagated through silu(g)*u and the scale;
* activation scales: |s - s_oracle| <= 1e-6 * s_oracle + (the same bound on the block max)/448;
* out: cosine >= 0.9999 and, element by element, |out - out_oracle| <= max(2e-2 *
  rms(out_oracle), one BF16 step at out_oracle); all-zero oracle rows must be exactly zero.
  The step term is the output's own final rounding: two FP32 sums that differ at all (the
  tensor core's block sums and the one-rounding promotion differ from the oracle's by
  design) can round to adjacent BF16 values, and one step of an output above 2.56 * rms is
  more than 2e-2 * rms. The counts of elements that needed it are printed.
"""
from __future__ import annotations

import os

import numpy as np
import torch
from scipy.special import expit

import oracle
from fp8_block_scaled_router_gb300 import _lib as L
from fp8_block_scaled_router_gb300 import inputs

NTHREADS = max(1, len(os.sched_getaffinity(0)))


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


class GpuMoE:
    """Device copies of one workload's parameters plus a workspace."""

    def __init__(self, x: inputs.MoEInputs, max_tokens: int):
        sh = x.shape
        self.x = x
        self.H, self.I, self.E, self.K = sh.hidden, sh.inter, sh.num_experts, sh.top_k
        self.shape = L.make_shape(self.H, self.I, self.E, self.K, max_tokens)
        self.w13, self.s13 = to_dev(x.w13), to_dev(x.s13)
        self.w2, self.s2 = to_dev(x.w2), to_dev(x.s2)
        self.router = to_dev(x.router_w)
        self.bias = None if x.bias is None else to_dev(x.bias)
        nb = L.moe_fp8_workspace_bytes(self.shape)
        assert nb > 0
        self.ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        L.moe_fp8_workspace_init(self.ws, self.shape)

    def route(self, hidden_d, M, renorm=True):
        ids = torch.empty((M, self.K), dtype=torch.int32, device="cuda")
        w = torch.empty((M, self.K), dtype=torch.float32, device="cuda")
        L.moe_route(hidden_d, self.router, self.bias, M, self.shape, renorm, ids, w)
        return ids, w

    def forward(self, hidden_d, ids_d, w_d, M, out=None):
        if out is None:
            out = torch.empty((M, self.H), dtype=torch.int16, device="cuda")
        L.moe_fp8_forward(hidden_d, ids_d, w_d, M, self.w13, self.s13, self.w2, self.s2, out,
                          self.ws, self.shape)
        return out

    def ws_arrays(self, M):
        v = L.moe_fp8_workspace_view(self.ws, self.shape)
        base = self.ws.data_ptr()
        R = M * self.K

        def sl(ptr, n, dtype):
            off = ptr - base
            nbytes = n * np.dtype(dtype).itemsize
            return self.ws[off: off + nbytes].cpu().numpy().view(dtype)

        return dict(qa=sl(v.qa, M * self.H, np.uint8).reshape(M, self.H),
                    sa=sl(v.sa, M * self.H // 128, np.float32).reshape(M, -1),
                    row_src=sl(v.row_src, R, np.int32), perm_row=sl(v.perm_row, R, np.int32),
                    act=sl(v.act, R * self.I, np.uint8).reshape(R, self.I),
                    act_scale=sl(v.act_scale, R * self.I // 128, np.float32).reshape(R, -1),
                    y=sl(v.y, R * self.H, np.float32).reshape(R, self.H),
                    offsets=sl(v.expert_offsets, self.E + 1, np.int32))

    def status(self):
        h = torch.zeros(1, dtype=torch.int32).pin_memory()
        L.moe_fp8_read_status(self.ws, h)
        torch.cuda.synchronize()
        return int(h[0])


# ---------------------------------------------------------------- comparisons
def bf16_f64(b):
    return inputs.bf16_bits_to_f32(b).astype(np.float64)


def bf16_step(b: np.ndarray) -> np.ndarray:
    """The spacing of BF16 values at |b| (8 significant bits; normal range)."""
    a = np.maximum(np.abs(b), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def out_bound_violations(a, b, rms, what):
    """Elements beyond max(2e-2 * rms, one BF16 step at the oracle's value); prints how many
    needed the step allowance."""
    d = np.abs(a - b)
    over_rms = d > 2e-2 * rms
    bad = over_rms & (d > bf16_step(b))
    if over_rms.any() and not bad.any():
        print(f"out [{what}]: {int(over_rms.sum())} element(s) beyond 2e-2*rms, each within one BF16 step "
              f"(|out| up to {float(np.max(np.abs(b[over_rms]))) / rms:.2f} rms)")
    return bad


def check_out(out_gpu: np.ndarray, out_orc: np.ndarray, what=""):
    a, b = bf16_f64(out_gpu), bf16_f64(out_orc)
    zero_rows = np.all(b == 0, axis=1)
    assert np.all(a[zero_rows] == 0), f"{what}: zero rows not exactly zero"
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    cos = 1.0 if na == 0 and nb == 0 else float(np.dot(a.ravel(), b.ravel()) / (na * nb))
    rms = float(np.sqrt(np.mean(b * b)))
    maxabs = float(np.max(np.abs(a - b)))
    assert cos >= 0.9999, f"{what}: cosine {cos}"
    bad = out_bound_violations(a, b, rms, what)
    assert not bad.any(), f"{what}: max|d| {maxabs} > max(2e-2 * rms {rms}, one BF16 step)"
    return cos, maxabs / max(rms, 1e-30)


def pair_act_from_ws(ws, M, K, I):
    """The GPU's activation codes and scales per routed pair [M][K][I] (expert-sorted rows
    mapped back through row_src; pairs that were not placed stay zero)."""
    R = len(ws["row_src"])
    q = np.zeros((M * K, I), np.uint8)
    sc = np.zeros((M * K, I // 128), np.float32)
    q[ws["row_src"]] = ws["act"][:R]
    sc[ws["row_src"]] = ws["act_scale"][:R]
    return q.reshape(M, K, I), sc.reshape(M, K, I // 128)


def check_out_given_act(out_gpu, out_orc, ws, dbg, ids, w, x, what="", down_combine=None):
    """The output bound with the contract's allowed activation-code differences accounted for.

    An activation code that check_act accepted one step away from the oracle's (its value
    next to a rounding boundary) changes the down projection of that routed row by design,
    by up to a few percent of rms(out). So: the whole output against the full oracle for
    cosine and exact zero rows; tokens whose activation codes all equal the oracle's against
    the full oracle for max|d| <= 2e-2 * rms(out_oracle); tokens with a differing code
    against the oracle's down projection and combine evaluated from the GPU's own codes and
    scales (oracle.down_combine, or the ``down_combine(qact, s2, ids, w)`` given), with the
    same bound."""
    M, K, I = ids.shape[0], ids.shape[1], x.shape.inter
    q_gpu, s_gpu = pair_act_from_ws(ws, M, K, I)
    valid = (ids >= 0) & (ids < x.shape.num_experts)
    diff = (q_gpu != dbg["qact"]) & ~(((q_gpu & 0x7F) == 0) & ((dbg["qact"] & 0x7F) == 0))
    diff &= valid[:, :, None]
    flip_tok = np.flatnonzero(diff.any(axis=(1, 2)))
    a, b = bf16_f64(out_gpu), bf16_f64(out_orc)
    zero_rows = np.all(b == 0, axis=1)
    assert np.all(a[zero_rows] == 0), f"{what}: zero rows not exactly zero"
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    cos = 1.0 if na == 0 and nb == 0 else float(np.dot(a.ravel(), b.ravel()) / (na * nb))
    rms = float(np.sqrt(np.mean(b * b)))
    assert cos >= 0.9999, f"{what}: cosine {cos}"
    keep = np.ones(M, bool)
    keep[flip_tok] = False
    err_keep = float(np.max(np.abs(a[keep] - b[keep]))) if keep.any() else 0.0
    err_flip_full = float(np.max(np.abs(a[flip_tok] - b[flip_tok]))) if len(flip_tok) else 0.0
    err_flip_cond = 0.0
    if len(flip_tok):
        if down_combine is None:
            cond = oracle.down_combine(q_gpu[flip_tok], s_gpu[flip_tok], ids[flip_tok], w[flip_tok], x.w2, x.s2,
                                       nthreads=NTHREADS)
        else:
            cond = down_combine(q_gpu[flip_tok], s_gpu[flip_tok], ids[flip_tok], w[flip_tok])
        err_flip_cond = float(np.max(np.abs(a[flip_tok] - bf16_f64(cond))))
    print(f"out [{what}]: cos {cos:.8f}, rms {rms:.4g}; {len(flip_tok)} of {M} tokens have a differing "
          f"activation code; max|d|/rms: other tokens {err_keep / rms:.3e}, those tokens vs the full oracle "
          f"{err_flip_full / rms:.3e}, vs the oracle from the GPU's codes {err_flip_cond / rms:.3e}")
    bad_keep = out_bound_violations(a[keep], b[keep], rms, what + ", tokens with the oracle's codes")
    assert not bad_keep.any(), f"{what}: max|d| {err_keep} > max(2e-2 * rms {rms}, one BF16 step)"
    if len(flip_tok):
        bad_flip = out_bound_violations(a[flip_tok], bf16_f64(cond), rms, what + ", given the GPU's codes")
        assert not bad_flip.any(), f"{what}: given the GPU's codes, max|d| {err_flip_cond} > 2e-2 * rms"
    return cos, max(err_keep, err_flip_cond) / max(rms, 1e-30)


_TAB = None


def e4m3_table64():
    global _TAB
    if _TAB is None:
        t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        _TAB = t
    return _TAB


def boundary_distance(v: np.ndarray) -> np.ndarray:
    """Distance from |v| to the nearest rounding midpoint of the E4M3 grid."""
    tab = e4m3_table64()
    mags = tab[:0x7F]                      # 0 .. 448 ascending
    mids = (mags[:-1] + mags[1:]) / 2
    a = np.minimum(np.abs(v), 448.0)
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    return np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))


def act_noise(dbg, t, j):
    """First-order bound (per unit of relative FP32 rounding) on the error of act = silu(g)*u
    from the rounding of g and u, whose promoted terms' magnitudes sum to gabs and uabs."""
    g = dbg["g"][t, j].astype(np.float64)
    u = dbg["u"][t, j].astype(np.float64)
    sg = expit(g)
    dg = np.abs(u * sg * (1 + g * (1 - sg)))
    du = np.abs(g * sg)
    return dg * dbg["gabs"][t, j] + du * dbg["uabs"][t, j]


# mismatch counts of every check_act call: (what, codes compared, mismatches inside the
# 1e-6 relative window, mismatches admitted only by the FP32 block-sum noise term)
ACT_COUNTS = []


def check_act(ws, dbg, K, what=""):
    """Compare expert-sorted GPU activation codes/scales with the oracle's per-pair ones.
    Returns (mismatches, compared codes, inside the 1e-6 window, only inside the noise term)."""
    row_src = ws["row_src"]
    R = len(row_src)
    t, j = row_src // K, row_src % K
    got_q, got_s = ws["act"][:R], ws["act_scale"][:R]
    exp_q, exp_s = dbg["qact"][t, j], dbg["s2"][t, j]
    act = dbg["act"][t, j].astype(np.float64)
    noise = act_noise(dbg, t, j)
    s_rep = np.repeat(exp_s.astype(np.float64), 128, axis=1)
    v = act / s_rep
    rel = 1e-6 * np.abs(v)
    window = rel + 5e-6 * noise / s_rep
    # +0 and -0 codes decode to the same value: not a mismatch
    mism = (got_q != exp_q) & ~(((got_q & 0x7F) == 0) & ((exp_q & 0x7F) == 0))
    n_rel = n_noise = 0
    if mism.any():
        dist = boundary_distance(v)
        near = dist <= window
        bad = mism & ~near
        assert not bad.any(), f"{what}: {int(bad.sum())} act codes differ away from a boundary"
        # inside the window: one code step at most (same sign, adjacent magnitude)
        step = np.abs(got_q[mism].astype(int) - exp_q[mism].astype(int))
        assert np.all(step == 1), what
        in_rel = mism & (dist <= rel)
        n_rel = int(in_rel.sum())
        n_noise = int(mism.sum()) - n_rel
    blk_noise = noise.reshape(R, -1, 128).max(-1)          # bound on |d amax| / 5e-6
    ds = np.abs(got_s.astype(np.float64) - exp_s)
    assert np.all(ds <= 1e-6 * exp_s + 5e-6 * blk_noise / 448.0 + 1e-45), f"{what}: act scales"
    ACT_COUNTS.append((what, int(mism.size), n_rel, n_noise))
    print(f"act codes [{what}]: {int(mism.size)} compared, {n_rel} mismatches within 1e-6 relative of a "
          f"boundary, {n_noise} admitted only by the block-sum noise term")
    return int(mism.sum()), int(mism.size), n_rel, n_noise


# Up to this many routed rows moe_fp8_forward runs every (token, slot) pair as its own unit
# (identity permutation); above it the pairs are sorted into expert-contiguous tiles.
PAIR_MAX_ROWS = 64


def check_permutation(ws, ids, E):
    """Pair mode: perm_row is the identity on valid pairs and -1 on skipped ones.
    Sorted mode: stable expert-sorted order -- row_src is a permutation of the valid pairs,
    increasing inside each expert segment, offsets match the histogram, perm_row inverts
    row_src."""
    flat = ids.ravel()
    valid = (flat >= 0) & (flat < E)
    if flat.size <= PAIR_MAX_ROWS:
        pr = ws["perm_row"][: flat.size]
        assert np.array_equal(pr, np.where(valid, np.arange(flat.size), -1))
        return
    counts = np.bincount(flat[valid], minlength=E)
    offs = ws["offsets"]
    assert offs[0] == 0 and np.array_equal(np.diff(offs), counts)
    R = int(valid.sum())
    rs = ws["row_src"][:R]
    assert sorted(rs.tolist()) == np.flatnonzero(valid).tolist()
    for e in range(E):
        seg = rs[offs[e]:offs[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    pr = ws["perm_row"][: flat.size]
    assert np.all(pr[~valid] == -1)
    assert np.array_equal(pr[rs], np.arange(R))


def oracle_route(x: inputs.MoEInputs, rows=None, renorm=True):
    hid = x.hidden if rows is None else x.hidden[rows]
    return oracle.route(hid, x.router_w, x.bias, x.shape.top_k, renormalize=renorm)


def oracle_forward(x, hidden, ids, w, debug=False):
    return oracle.moe_forward(hidden, ids, w, x.w13, x.s13, x.w2, x.s2, debug=debug,
                              nthreads=NTHREADS)
