"""Seeded synthetic inputs for the routed FP8 MoE FFN (shared by the tests, the bench and
the oracle's callers).

This module draws random numbers and packs them into the library's layouts. It holds none
of the layer's own arithmetic (no routing, no requantisation, no GEMM): the weights are
quantised here the way an FP8 checkpoint is prepared (one FP32 scale per 128x128 block,
scale = block amax / 448, codes from torch's ``float8_e4m3fn`` cast), which is input
preparation, not the hot path.

Workload recipes (shapes follow the netra-kernel pages' Qwen3.6 FP8 MoE regimes and the
amd-kernels wide-expert shape token h6144_i768_e128_top4):

* hidden states BF16 ~ N(0, 1) (round to nearest even);
* router weights BF16 [H][E] ~ N(0, 0.02), except prefill, where N(0, 1/sqrt(H)) makes the
  logits ~ N(0, 1);
* w13 [E][2I][H] and w2 [E][H][I] ~ N(0, 0.02) in FP32, quantised per 128x128 block;
* skewed verify: an FP32 logit bias of +3.0 on experts 0..3;
* Zipf prefill: each token draws K distinct experts with p(e) proportional to (e+1)^-1.1,
  without replacement (Gumbel top-k), and Dirichlet(1) weights;
* MXFP4 expert weights (the h6144/i768/e128/top-4 shape token): the same N(0, 0.02) draws,
  quantised per 32 consecutive K elements with scale 2^(floor(log2(amax)) - 2) and
  round-to-nearest-even E2M1 codes saturating at 6 (OCP microscaling);
* the un-normalised hidden in front of an RMSNorm (the residual stream): each row
  N(0, sigma_t^2) with sigma_t log-uniform in [2^-4, 2^4], and 4 outlier channels (drawn
  once per seed) scaled by 16; the norm's weight BF16 ~ 1 + N(0, 0.1^2).

Every stream is ``numpy.random.default_rng([seed, stream])`` (PCG64) so that each tensor
is independent of the order in which the others are drawn.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# stream ids for default_rng([seed, stream])
_S_HIDDEN, _S_ROUTER, _S_W13, _S_W2, _S_IDS, _S_WTS = 1, 2, 3, 4, 5, 6
_S_RESID, _S_GAMMA = 7, 8


@dataclasses.dataclass(frozen=True)
class Shape:
    hidden: int       # H
    inter: int        # I (per-expert intermediate)
    num_experts: int  # E
    top_k: int        # K


# Named workloads: shape, tokens per launch, router std, seed.
CONFIGS = {
    "tiny": dict(shape=Shape(256, 128, 8, 2), M=4, router_std=0.02, seed=0),
    "decode": dict(shape=Shape(2048, 768, 128, 8), M=1, router_std=0.02, seed=1, tokens=10000),
    "verify": dict(shape=Shape(2048, 768, 128, 8), M=12, router_std=0.02, seed=2),
    "verify_skewed": dict(shape=Shape(2048, 768, 128, 8), M=12, router_std=0.02, seed=2,
                          hot_bias=3.0, hot_experts=(0, 1, 2, 3)),
    "wide": dict(shape=Shape(6144, 768, 128, 4), M=64, router_std=0.02, seed=3,
                 sweep=(1, 2, 4, 8, 16, 32, 64)),
    "prefill": dict(shape=Shape(2048, 768, 128, 8), M=4096, router_std=None, seed=4),
    "prefill_zipf": dict(shape=Shape(2048, 768, 128, 8), M=4096, router_std=None, seed=5,
                         zipf=1.1),
    # edges of the supported shape set (parity tests only): the largest hidden and
    # intermediate sizes, the most experts with the largest top-k, and top-1
    "max_dims": dict(shape=Shape(8192, 4096, 8, 8), M=16, router_std=0.02, seed=6),
    "many_experts": dict(shape=Shape(256, 128, 256, 16), M=24, router_std=0.02, seed=7),
    "top1": dict(shape=Shape(2048, 768, 16, 1), M=100, router_std=0.02, seed=8),
}


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 (torch's round-to-nearest-even cast), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def hidden_states(seed: int, M: int, H: int, zero_rows: Optional[np.ndarray] = None) -> np.ndarray:
    x = rng(seed, _S_HIDDEN).standard_normal((M, H), dtype=np.float32)
    if zero_rows is not None:
        x[zero_rows] = 0.0
    return to_bf16_bits(x)


def router_weights(seed: int, H: int, E: int, std: Optional[float]) -> np.ndarray:
    if std is None:
        std = 1.0 / np.sqrt(H)
    return to_bf16_bits(rng(seed, _S_ROUTER).standard_normal((H, E), dtype=np.float32) * np.float32(std))


def quantise_weight_blocks(w: np.ndarray):
    """One expert matrix [N][Kd] FP32 -> (E4M3 codes uint8 [N][Kd], FP32 scales [N/128][Kd/128])."""
    N, Kd = w.shape
    blocks = w.reshape(N // 128, 128, Kd // 128, 128)
    amax = np.abs(blocks).max(axis=(1, 3)).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    scaled = (blocks / scale[:, None, :, None]).astype(np.float32).reshape(N, Kd)
    codes = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def expert_weights(seed: int, stream: int, E: int, N: int, Kd: int, std: float = 0.02):
    """[E][N][Kd] E4M3 codes and [E][N/128][Kd/128] FP32 scales, drawn one expert at a time."""
    g = rng(seed, stream)
    codes = np.empty((E, N, Kd), np.uint8)
    scales = np.empty((E, N // 128, Kd // 128), np.float32)
    for e in range(E):
        w = g.standard_normal((N, Kd), dtype=np.float32) * np.float32(std)
        codes[e], scales[e] = quantise_weight_blocks(w)
    return codes, scales


@dataclasses.dataclass
class MoEInputs:
    shape: Shape
    M: int
    hidden: np.ndarray          # uint16 (BF16) [M][H]
    router_w: np.ndarray        # uint16 (BF16) [H][E]
    bias: Optional[np.ndarray]  # f32 [E] or None
    w13: np.ndarray             # uint8 (E4M3) [E][2I][H]
    s13: np.ndarray             # f32 [E][2I/128][H/128]
    w2: np.ndarray              # uint8 (E4M3) [E][H][I]
    s2: np.ndarray              # f32 [E][H/128][I/128]
    ids: Optional[np.ndarray] = None      # int32 [M][K] when routing is given (Zipf)
    weights: Optional[np.ndarray] = None  # f32 [M][K] when routing is given


def zipf_routing(seed: int, M: int, E: int, K: int, a: float):
    """K distinct experts per token, p(e) ~ (e+1)^-a, without replacement; Dirichlet weights."""
    g = rng(seed, _S_IDS)
    logp = -a * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logp[None, :] + g.gumbel(size=(M, E))
    ids = np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    wts = rng(seed, _S_WTS).dirichlet(np.ones(K), size=M).astype(np.float32)
    return ids, wts


def make(name: str, M: Optional[int] = None, E: Optional[int] = None, tokens: Optional[int] = None,
         zero_rows: Optional[np.ndarray] = None) -> MoEInputs:
    """Build a named workload. ``M`` overrides the token count, ``tokens`` the number of
    hidden rows drawn (decode draws many rows, one per launch), ``E`` the expert count
    (to shrink a config for a fast test; the per-expert shapes are unchanged)."""
    c = CONFIGS[name]
    sh: Shape = c["shape"]
    if E is not None:
        sh = dataclasses.replace(sh, num_experts=E)
    M = c["M"] if M is None else M
    rows = M if tokens is None else tokens
    seed = c["seed"]
    H, I, Ex, K = sh.hidden, sh.inter, sh.num_experts, sh.top_k
    hidden = hidden_states(seed, rows, H, zero_rows)
    router_w = router_weights(seed, H, Ex, c["router_std"])
    bias = None
    if "hot_bias" in c:
        bias = np.zeros(Ex, np.float32)
        bias[list(c["hot_experts"])] = np.float32(c["hot_bias"])
    w13, s13 = expert_weights(seed, _S_W13, Ex, 2 * I, H)
    w2, s2 = expert_weights(seed, _S_W2, Ex, H, I)
    ids = wts = None
    if "zipf" in c:
        ids, wts = zipf_routing(seed, rows, Ex, K, c["zipf"])
    return MoEInputs(sh, M, hidden, router_w, bias, w13, s13, w2, s2, ids, wts)


# ---- MXFP4 weights (OCP microscaling: E2M1 codes, one UE8M0 scale per 32 elements) -------
# The magnitudes of E2M1 codes 0..7 (the format's value table; the sign is bit 3).
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


_E2M1_MIDPOINTS = ((E2M1_MAGNITUDES[:-1] + E2M1_MAGNITUDES[1:]) / 2).astype(np.float32)  # exact in FP32


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value, ties to the even code, saturating at +-6; uint8 codes.
    (FP32 input: every midpoint between E2M1 values is exact in FP32.)"""
    x = np.asarray(x, np.float32)
    a = np.abs(x)
    mag = np.searchsorted(_E2M1_MIDPOINTS, a, side="left").astype(np.uint8)  # midpoints below a
    at_mid = a == _E2M1_MIDPOINTS[np.minimum(mag, 6)]
    mag += (at_mid & (mag < 7) & ((mag & 1) == 1)).astype(np.uint8)         # halfway: the even code
    return mag | (np.signbit(x).astype(np.uint8) << 3)


def mx_quantise_blocks(w: np.ndarray):
    """One expert matrix [N][Kd] FP32 -> (codes [N][Kd/2], two per byte, the lower K index in
    the low nibble; UE8M0 scales [N][Kd/32]). Scale = 2^(floor(log2(block amax)) - 2) (the
    largest E2M1 exponent is 2); an all-zero block takes 2^-127. The codes are e2m1_encode of
    the scaled values (computed here with torch's CPU kernels, which run on every core)."""
    N, Kd = w.shape
    mids = torch.from_numpy(_E2M1_MIDPOINTS)
    b = torch.from_numpy(np.ascontiguousarray(w, np.float32)).reshape(N, Kd // 32, 32)
    amax = b.abs().amax(dim=-1)
    _, e2 = torch.frexp(amax)  # amax = f * 2^e2 with f in [0.5, 1): floor(log2(amax)) = e2 - 1
    ex = torch.where(amax > 0, e2 - 3, torch.full_like(e2, -127)).clamp(-127, 127)
    scaled = b * torch.ldexp(torch.ones_like(amax), -ex)[..., None]  # exact: a power of two
    a = scaled.abs()
    mag = torch.bucketize(a, mids, right=False).to(torch.uint8)  # midpoints below a
    at_mid = a == mids[mag.clamp(max=6).long()]
    mag = mag + (at_mid & (mag < 7) & ((mag & 1) == 1)).to(torch.uint8)  # halfway: the even code
    codes = (mag | (torch.signbit(scaled).to(torch.uint8) << 3)).reshape(N, Kd)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.numpy().astype(np.uint8), (ex + 127).to(torch.uint8).numpy()


def mx_expert_weights(seed: int, stream: int, E: int, N: int, Kd: int, std: float = 0.02):
    """[E][N][Kd/2] packed E2M1 codes and [E][N][Kd/32] UE8M0 scales, one expert at a time."""
    g = rng(seed, stream)
    codes = np.empty((E, N, Kd // 2), np.uint8)
    scales = np.empty((E, N, Kd // 32), np.uint8)
    for e in range(E):
        codes[e], scales[e] = mx_quantise_blocks(g.standard_normal((N, Kd), dtype=np.float32) * np.float32(std))
    return codes, scales


MX_CONFIGS = {
    # the amd-kernels MXFP4 shape token h6144_i768_e128_top4, token count a runtime argument
    "wide_mxfp4": dict(shape=Shape(6144, 768, 128, 4), M=64, router_std=0.02, seed=9),
    "tiny_mxfp4": dict(shape=Shape(256, 128, 8, 2), M=4, router_std=0.02, seed=10),
}


def make_mx(name: str, M: Optional[int] = None, tokens: Optional[int] = None, E: Optional[int] = None) -> "MoEInputs":
    """A named MXFP4 workload: w13 / w2 hold packed E2M1 codes, s13 / s2 UE8M0 scales. ``E``
    overrides the expert count (a smaller draw for a fast test; the per-expert shapes are
    unchanged)."""
    c = MX_CONFIGS[name]
    sh: Shape = c["shape"]
    if E is not None:
        sh = dataclasses.replace(sh, num_experts=E)
    M = c["M"] if M is None else M
    rows = M if tokens is None else tokens
    seed = c["seed"]
    H, I, E = sh.hidden, sh.inter, sh.num_experts
    hidden = hidden_states(seed, rows, H)
    router_w = router_weights(seed, H, E, c["router_std"])
    w13, s13 = mx_expert_weights(seed, _S_W13, E, 2 * I, H)
    w2, s2 = mx_expert_weights(seed, _S_W2, E, H, I)
    return MoEInputs(sh, M, hidden, router_w, None, w13, s13, w2, s2, None, None)


def residual_states(seed: int, M: int, H: int, zero_rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Un-normalised BF16 rows [M][H] (uint16 bits) for the RMSNorm in front of the layer."""
    g = rng(seed, _S_RESID)
    sigma = np.exp2(g.uniform(-4.0, 4.0, size=(M, 1))).astype(np.float32)
    x = g.standard_normal((M, H), dtype=np.float32) * sigma
    outliers = g.choice(H, size=4, replace=False)
    x[:, outliers] *= np.float32(16.0)
    if zero_rows is not None:
        x[zero_rows] = 0.0
    return to_bf16_bits(x)


def norm_weight(seed: int, H: int) -> np.ndarray:
    """The RMSNorm weight, BF16 [H] (uint16 bits)."""
    return to_bf16_bits(1.0 + 0.1 * rng(seed, _S_GAMMA).standard_normal(H, dtype=np.float32))


def wide_padding_rows(M: int) -> np.ndarray:
    """Rows of zeros at the end of a wide-sweep batch, as CUDA-graph padding leaves them."""
    return np.arange(M - M // 4, M)
