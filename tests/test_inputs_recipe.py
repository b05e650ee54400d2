"""The synthetic input recipe (no GPU): seeded and reproducible, and shaped as stated -- hidden
~N(0,1) in BF16; router N(0, 0.02), or N(0, 1/sqrt(H)) for prefill so that logits ~N(0,1);
expert weights quantised per 128x128 block with scale amax/448, so every block reaches the
E4M3 maximum; the skewed verify bias; Zipf(1.1) expert ranks with distinct ids and Dirichlet
weights; zero padding rows at the end of a wide batch."""
import numpy as np
import torch

from fp8_block_scaled_router_gb300 import inputs


def dec(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_workloads_are_reproducible():
    a, b = inputs.make("tiny"), inputs.make("tiny")
    for f in ("hidden", "router_w", "w13", "s13", "w2", "s2"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_seeds_and_streams_are_independent():
    h1 = inputs.hidden_states(1, 4, 256)
    h2 = inputs.hidden_states(2, 4, 256)
    assert not np.array_equal(h1, h2)
    w13, _ = inputs.expert_weights(0, inputs._S_W13, 1, 128, 128)
    w2, _ = inputs.expert_weights(0, inputs._S_W2, 1, 128, 128)
    assert not np.array_equal(w13, w2)


def test_every_weight_block_reaches_the_e4m3_maximum():
    codes, scales = inputs.expert_weights(3, inputs._S_W13, 2, 256, 384)
    v = np.abs(dec(codes)).reshape(2, 2, 128, 3, 128)
    assert np.all(v.max(axis=(2, 4)) == 448.0)
    assert np.all(scales > 0)
    # dequantised block maximum = the block's FP32 amax = 448 * scale
    g = inputs.rng(3, inputs._S_W13)
    w0 = g.standard_normal((256, 384), dtype=np.float32) * np.float32(0.02)
    amax = np.abs(w0).reshape(2, 128, 3, 128).max(axis=(1, 3))
    assert np.array_equal(scales[0], (amax / np.float32(448)).astype(np.float32))


def test_hidden_is_standard_normal_bf16():
    h = inputs.bf16_bits_to_f32(inputs.hidden_states(4, 64, 2048)).astype(np.float64)
    assert abs(h.mean()) < 0.01 and abs(h.std() - 1.0) < 0.01


def test_prefill_router_gives_unit_logits():
    H, E = 2048, 128
    x = inputs.bf16_bits_to_f32(inputs.hidden_states(4, 256, H)).astype(np.float64)
    w = inputs.bf16_bits_to_f32(inputs.router_weights(4, H, E, None)).astype(np.float64)
    logits = x @ w
    assert abs(logits.std() - 1.0) < 0.05
    wd = inputs.bf16_bits_to_f32(inputs.router_weights(1, H, E, 0.02)).astype(np.float64)
    assert abs(wd.std() - 0.02) < 0.001


def test_skewed_verify_bias():
    c = inputs.CONFIGS["verify_skewed"]
    assert c["hot_bias"] == 3.0 and tuple(c["hot_experts"]) == (0, 1, 2, 3)


def test_zipf_routing():
    M, E, K = 4096, 128, 8
    ids, wts = inputs.zipf_routing(5, M, E, K, 1.1)
    assert ids.shape == (M, K) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(r)) == K for r in ids.tolist())
    assert np.all(wts > 0) and np.allclose(wts.sum(1), 1.0, atol=1e-5)
    counts = np.bincount(ids.ravel(), minlength=E)
    # the load falls with the expert's rank: the head expert is busiest, the tail lightest
    assert counts[0] == counts.max() and counts[:8].mean() > 2 * counts[-32:].mean()


def test_wide_padding_rows_are_zero():
    rows = inputs.wide_padding_rows(64)
    assert np.array_equal(rows, np.arange(48, 64))
    h = inputs.hidden_states(3, 64, 256, zero_rows=rows)
    assert np.all(h[48:] == 0) and np.all(np.any(h[:48] != 0, axis=1))
