"""Pins for the oracle's RMSNorm (the normalisation in front of the routed layer).

The netra-kernel lab's gfx950 layout lists normalisation and quantisation fusions, and the
Qwen3.6 RMSNorm work sits in front of the MoE block; the pages give no epsilon and no weight
convention, so the oracle takes the plain definition y = bf16(x * gamma / sqrt(mean(x^2) +
eps)) with eps and gamma from the caller. These pins hold it to what the mathematics fixes:
a float64 evaluation of that closed form (to one BF16 step, nearly always exact), torch's
own rms_norm, exact special cases (powers of two, constant, zero and one-hot rows) and the
scale invariance of the definition at eps = 0.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

U = 2.0 ** -24


def f32(b):
    return inputs.bf16_bits_to_f32(b)


def closed_form(x, g, eps):
    xd, gd = f32(x).astype(np.float64), f32(g).astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + eps)
    return xd * r * gd[None, :], r[:, 0]


def bf16_step(v):
    """The spacing of BF16 values at |v| (8 significant bits)."""
    a = np.maximum(np.abs(v), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("M,H,eps", [(64, 2048, 1e-6), (16, 6144, 1e-6), (32, 256, 1e-2), (8, 8192, 1e-5)])
def test_rmsnorm_matches_float64_closed_form(oracle_mod, M, H, eps):
    x = inputs.residual_states(21, M, H)
    g = inputs.norm_weight(21, H)
    y, r = oracle_mod.rmsnorm(x, g, eps, want_rstd=True)
    ref, rref = closed_form(x, g, eps)
    # r: the chunk chains' relative error is below (128 + H/128) u, the rest a few roundings
    assert np.all(np.abs(r - rref) <= (0.5 * (128 + H // 128) + 4) * U * rref)
    yv = f32(y).astype(np.float64)
    assert np.all(np.abs(yv - ref) <= bf16_step(ref))  # within one BF16 step everywhere
    exact = f32(inputs.to_bf16_bits(ref.astype(np.float32)))
    assert np.mean(yv == exact) >= 0.99                 # and the nearest BF16 almost always


def test_rmsnorm_small_rows_feel_eps(oracle_mod):
    # rows with mean(x^2) ~ eps: a dropped or misplaced eps moves y by a large factor
    M, H, eps = 16, 1024, 1e-2
    x = inputs.to_bf16_bits(np.full((M, H), 0.1, np.float32) * np.linspace(0.5, 2.0, M, dtype=np.float32)[:, None])
    g = inputs.norm_weight(22, H)
    y = oracle_mod.rmsnorm(x, g, eps)
    ref, _ = closed_form(x, g, eps)
    assert np.all(np.abs(f32(y) - ref) <= bf16_step(ref))


def test_rmsnorm_matches_torch(oracle_mod):
    M, H, eps = 48, 2048, 1e-6
    x = inputs.residual_states(23, M, H)
    g = inputs.norm_weight(23, H)
    y = f32(oracle_mod.rmsnorm(x, g, eps)).astype(np.float64)
    xt = torch.from_numpy(f32(x))
    gt = torch.from_numpy(f32(g))
    ref = torch.nn.functional.rms_norm(xt.double(), (H,), weight=gt.double(), eps=eps).numpy()
    assert np.all(np.abs(y - ref) <= bf16_step(ref))
    t32 = torch.nn.functional.rms_norm(xt, (H,), weight=gt, eps=eps).to(torch.bfloat16).float().numpy()
    assert np.mean(y == t32) >= 0.98  # torch's FP32 order differs from the chunk chains


@pytest.mark.parametrize("H", [256, 2048, 6144])
def test_rmsnorm_constant_rows_are_exact(oracle_mod, H):
    # c a power of two: every square and partial sum is exact, mean = c^2, r = 1/|c|
    c = np.array([2.0 ** -6, -0.5, 1.0, 8.0, -64.0], np.float32)
    x = inputs.to_bf16_bits(np.repeat(c[:, None], H, axis=1))
    g = inputs.to_bf16_bits(np.ones(H, np.float32))
    y, r = oracle_mod.rmsnorm(x, g, 0.0, want_rstd=True)
    assert np.array_equal(r, (1.0 / np.abs(c)).astype(np.float32))
    assert np.array_equal(f32(y), np.repeat(np.sign(c)[:, None], H, axis=1).astype(np.float32))
    gw = inputs.norm_weight(24, H)
    y2 = oracle_mod.rmsnorm(x, gw, 0.0)
    assert np.array_equal(f32(y2), np.sign(c)[:, None] * f32(gw)[None, :])


def test_rmsnorm_zero_row_and_one_hot(oracle_mod):
    H, eps = 2048, 1e-6
    x = np.zeros((3, H), np.float32)
    x[1, 77] = 3.0
    x[2, 2047] = -0.25
    xb = inputs.to_bf16_bits(x)
    g = inputs.norm_weight(25, H)
    y, r = oracle_mod.rmsnorm(xb, g, eps, want_rstd=True)
    assert np.all(f32(y[0]) == 0.0) and r[0] == np.float32(1.0 / np.sqrt(np.float32(eps)))
    ref, rref = closed_form(xb, g, eps)
    for t, k in ((1, 77), (2, 2047)):
        assert abs(f32(y[t, k]) - ref[t, k]) <= bf16_step(ref[t, k])  # ~ sign * sqrt(H) * g_k
        assert np.count_nonzero(y[t]) == 1


def test_rmsnorm_is_scale_invariant_at_zero_eps(oracle_mod):
    # powers of two scale every step exactly: y(2^k x) == y(x) bit for bit
    M, H = 24, 2048
    x = inputs.residual_states(26, M, H)
    g = inputs.norm_weight(26, H)
    y0 = oracle_mod.rmsnorm(x, g, 0.0)
    for k in (-3, 2, 5):
        xs = inputs.to_bf16_bits(f32(x) * np.float32(2.0 ** k))
        assert np.array_equal(oracle_mod.rmsnorm(xs, g, 0.0), y0)


def test_rmsnorm_rejects_bad_sizes(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.rmsnorm(np.zeros((2, 200), np.uint16), np.zeros(200, np.uint16), 1e-6)
