"""Pins for the oracle's FP8 E4M3 codec and its per-128 quantiser.

The codec is pinned to the E4M3 ("fn") format definition and, independently, to torch's
``float8_e4m3fn`` casts (a library routine that shares nothing with the oracle). Format
used by the pages: "NetraRuntime/netra-kernel" lab README, "Supported targets" table
(FP8 E4M3 with 128x128 block scales).
"""
import numpy as np
import pytest
import torch


def torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def torch_encode(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_table_matches_torch_decode(oracle_mod):
    tab = oracle_mod.e4m3_table()
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(tab), nan)
    assert np.array_equal(tab[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_table_format_landmarks(oracle_mod):
    tab = oracle_mod.e4m3_table()
    assert np.flatnonzero(np.isnan(tab)).tolist() == [0x7F, 0xFF]
    assert tab[0x7E] == 448.0 and np.nanmax(tab) == 448.0
    assert tab[0xFE] == -448.0
    assert tab[0x01] == 2.0 ** -9 and tab[0x07] == 7 * 2.0 ** -9      # subnormals m * 2^-9
    assert tab[0x08] == 2.0 ** -6                                       # smallest normal
    assert tab[0x38] == 1.0                                             # exponent field 7 = bias
    assert tab[0x00] == 0.0 and np.signbit(tab[0x80])
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)                                     # strictly monotone
    assert np.array_equal(tab[0x80:0xFF], -tab[0x00:0x7F])


def test_every_code_round_trips(oracle_mod):
    tab = oracle_mod.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle_mod.e4m3_encode(tab[codes]), codes)


def test_midpoints_round_to_even(oracle_mod):
    tab = oracle_mod.e4m3_table().astype(np.float64)
    lo = np.arange(0, 0x7E)
    mids = ((tab[lo] + tab[lo + 1]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (tab[lo] + tab[lo + 1]) / 2)  # exact in f32
    q = oracle_mod.e4m3_encode(mids)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(q, expect)
    # one FP32 ulp either side of each midpoint goes to the nearer code
    above = np.nextafter(mids, np.float32(np.inf))
    below = np.nextafter(mids, np.float32(-np.inf))
    assert np.array_equal(oracle_mod.e4m3_encode(above), (lo + 1).astype(np.uint8))
    assert np.array_equal(oracle_mod.e4m3_encode(below), lo.astype(np.uint8))
    # negative side mirrors with the sign bit
    assert np.array_equal(oracle_mod.e4m3_encode(-mids), expect | 0x80)


def test_saturation_nan_and_signed_zero(oracle_mod):
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(oracle_mod.e4m3_encode(big) == 0x7E)
    assert np.all(oracle_mod.e4m3_encode(-big) == 0xFE)
    assert oracle_mod.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    assert oracle_mod.e4m3_encode(np.array([0.0], np.float32))[0] == 0x00
    assert oracle_mod.e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80
    # below half the smallest subnormal: rounds to a signed zero
    tiny = np.float32(2.0 ** -11)
    assert oracle_mod.e4m3_encode(np.array([tiny, -tiny], np.float32)).tolist() == [0x00, 0x80]


@pytest.mark.parametrize("seed", [0, 1])
def test_encoder_matches_torch_cast_in_range(oracle_mod, seed):
    g = np.random.default_rng(seed)
    # log-uniform magnitudes spanning subnormals to the top of the range, both signs
    mag = np.exp(g.uniform(np.log(2.0 ** -12), np.log(447.9), 200_000)).astype(np.float32)
    x = np.where(g.random(mag.size) < 0.5, -mag, mag).astype(np.float32)
    assert np.array_equal(oracle_mod.e4m3_encode(x), torch_encode(x))


def test_encoder_matches_torch_on_strided_bit_sweep(oracle_mod):
    bits = np.arange(0, 2 ** 32, 4099, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    keep = np.isfinite(x) & (np.abs(x) < 448.0)
    x = x[keep]
    assert np.array_equal(oracle_mod.e4m3_encode(x), torch_encode(x))


def test_quantiser_zero_group(oracle_mod):
    q, s = oracle_mod.quantise(np.zeros((3, 256), np.float32))
    assert np.all(q == 0) and np.all(s == 1.0)


def test_quantiser_scale_and_error_bound(oracle_mod):
    g = np.random.default_rng(7)
    x = (g.standard_normal((64, 512)) * np.exp(g.uniform(-6, 6, (64, 1)))).astype(np.float32)
    q, s = oracle_mod.quantise(x)
    blocks = x.reshape(64, 4, 128)
    amax = np.abs(blocks).max(axis=2)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    # the element holding the group maximum encodes to +-448
    arg = np.abs(blocks).argmax(axis=2)
    qb = q.reshape(64, 4, 128)
    top = np.take_along_axis(qb, arg[..., None], axis=2)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    # dequantised values sit within half an E4M3 spacing (relative 2^-4) of the inputs,
    # or within half the subnormal step 2^-10 (times the scale) near zero
    deq = torch_decode(q).reshape(64, 4, 128) * s[..., None]
    err = np.abs(deq - blocks)
    allow = np.maximum(np.abs(blocks) * 2.0 ** -4, s[..., None] * 2.0 ** -10) * 1.0001
    assert np.all(err <= allow)


def test_block_dot_is_exact(oracle_mod):
    """The 128-term FP8 block sum equals an exact integer recomputation, rounded once."""
    g = np.random.default_rng(3)
    tab = torch_decode(np.arange(256, dtype=np.uint8))
    finite = np.flatnonzero(np.isfinite(tab)).astype(np.uint8)
    for _ in range(200):
        a = g.choice(finite, 128)
        w = g.choice(finite, 128)
        ia = np.round(tab[a].astype(np.float64) * 512).astype(np.int64)  # exact: m * 2^-9
        iw = np.round(tab[w].astype(np.float64) * 512).astype(np.int64)
        exact = int(np.dot(ia, iw))                       # units of 2^-18, |.| < 2^43
        ref = np.float32(exact / 2.0 ** 18)               # one rounding (exact < 2^53 in f64)
        got = np.float32(oracle_mod.block_dot(a, w))
        assert got == ref
