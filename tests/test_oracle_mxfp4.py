"""Pins for the oracle's MXFP4 weight variant (the amd-kernels h6144_i768_e128_top4 MXFP4
shape token; the kernel-lab README's gfx1151 MXFP4 target, validated against FP64
dequantised-MXFP4 references).

MXFP4 is OCP microscaling with FP4 elements: E2M1 codes and one UE8M0 scale (2^(e-127)) per
32 consecutive elements along K. The pins hold the oracle to:
* the E2M1 value table of the format and torch's UE8M0 (float8_e8m0fnu) decoding;
* the input preparation's encoder against brute force, and the block quantiser's range;
* a float64 dequantised reference within a rigorous rounding bound (one row, gate/up,
  down, and the whole layer through the FP8 layer's combine), closed forms with exact
  small-integer data, and brute force over every expert.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_router_gb300 import inputs

U = 2.0 ** -24
# the E2M1 value table of the format (sign, 2 exponent bits with bias 1, 1 mantissa bit)
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1_dec(codes):
    c = np.asarray(codes, np.int64)
    mag = np.array(E2M1)[c & 7]
    return np.where(c & 8, -mag, mag)


def unpack(q):
    """[..., K/2] packed -> [..., K] codes (lower K index in the low nibble)."""
    q = np.asarray(q, np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = q & 15
    out[..., 1::2] = q >> 4
    return out


def deq_mx(q, s):
    """codes [..., K/2], UE8M0 scales [..., K/32] -> float64 [..., K]."""
    sc = torch.from_numpy(np.ascontiguousarray(s, np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    return e2m1_dec(unpack(q)) * np.repeat(sc, 32, -1)


def dec_e4m3(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e2m1_table_is_the_format_table(oracle_mod):
    t = oracle_mod.e2m1_table()
    assert t[:8].tolist() == E2M1
    assert t[8:].tolist() == [-v for v in E2M1] and np.all(np.signbit(t[8:]))


def test_ue8m0_decode_matches_torch(oracle_mod):
    e = np.arange(256, dtype=np.uint8)
    got = oracle_mod.ue8m0_decode(e)
    ref = torch.from_numpy(e).view(torch.float8_e8m0fnu).to(torch.float32).numpy()
    assert np.array_equal(got[:255], ref[:255]) and np.isnan(got[255]) and np.isnan(ref[255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_e2m1_encoder_against_brute_force():
    g = np.random.default_rng(3)
    x = np.concatenate([g.uniform(-8, 8, 20000), np.array(E2M1) + 0.0, -np.array(E2M1),
                        (np.array(E2M1[:-1]) + np.array(E2M1[1:])) / 2, [7.0, 100.0, -1e9, -0.0]]).astype(np.float32)
    got = inputs.e2m1_encode(x)
    vals = np.array(E2M1)
    for xi, gi in zip(x.astype(np.float64), got):
        a = min(abs(xi), 6.0)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else best[best % 2 == 0][0]  # halfway: the even code
        assert gi == (code | (8 if np.signbit(xi) else 0)), (xi, gi, code)


def test_block_quantiser_range_and_error():
    g = np.random.default_rng(4)
    w = (g.standard_normal((64, 512)) * 0.02).astype(np.float32)
    w[3, :32] = 0.0  # an all-zero block
    q, s = inputs.mx_quantise_blocks(w)
    assert q.shape == (64, 256) and s.shape == (64, 16)
    back = deq_mx(q, s)
    blocks = np.abs(w.reshape(64, 16, 32)).max(-1)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    ratio = np.where(blocks > 0, blocks / scale, 4.0)
    assert np.all((ratio >= 4.0) & (ratio < 8.0))  # scale = 2^(floor(log2 amax) - 2)
    assert s[3, 0] == 0 and np.all(q[3, :16] == 0)
    # within half a step of the E2M1 grid, or saturated at 6 * scale (amax / scale in [6, 8))
    err = np.abs(back - w.astype(np.float64))
    step = np.repeat(scale, 32, -1)
    sat = np.abs(w) >= 6.0 * step
    assert np.all(err[~sat] <= step[~sat] * 1.0 + 1e-30)
    assert np.all(np.abs(back[sat]) == 6.0 * step[sat])


def _row_case(seed, K=512):
    g = np.random.default_rng(seed)
    a = g.integers(0, 256, K).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38  # no NaN codes
    sa = np.ldexp(1.0, g.integers(-4, 4, K // 128)).astype(np.float32) * np.float32(1.25)
    wq = g.integers(0, 256, K // 2).astype(np.uint8)
    ws = g.integers(110, 140, K // 32).astype(np.uint8)
    return a, sa, wq, ws


@pytest.mark.parametrize("seed", range(6))
def test_mx_row_within_float64_bound(oracle_mod, seed):
    a, sa, wq, ws = _row_case(seed)
    got = oracle_mod.mx_row(a, sa, wq, ws)
    av = dec_e4m3(a) * np.repeat(sa.astype(np.float64), 128)
    wv = deq_mx(wq, ws)
    ref = float(av @ wv)
    # per 32-block one rounding (exact dot), 4 sub-block adds and the scale multiply per
    # 128-block, one multiply and one add per block in the chain
    bound = (1 + 4 + 2 + len(sa) + 2) * U * float(np.abs(av) @ np.abs(wv)) * 1.01
    assert abs(got - ref) <= bound


def test_mx_row_closed_forms(oracle_mod):
    K = 256
    a = np.full(K, 0x38, np.uint8)                      # 1.0
    sa = np.ones(K // 128, np.float32)
    wq = np.full(K // 2, 0x22, np.uint8)                # E2M1 code 2 (1.0) twice
    ws = np.full(K // 32, 127, np.uint8)                # 2^0
    assert oracle_mod.mx_row(a, sa, wq, ws) == 256.0
    ws = np.tile(np.array([127, 128, 129, 130], np.uint8), K // 128)  # sub-block scales 1, 2, 4, 8
    assert oracle_mod.mx_row(a, sa, wq, ws) == 2 * 32 * (1 + 2 + 4 + 8)
    wq = np.full(K // 2, 0xF7, np.uint8)                # codes 7 (6.0) and 15 (-6.0): cancel
    assert oracle_mod.mx_row(a, sa, wq, np.full(K // 32, 127, np.uint8)) == 0.0
    sa = np.array([0.5, 3.0], np.float32)
    wq = np.full(K // 2, 0x33, np.uint8)                # 1.5
    assert oracle_mod.mx_row(a, sa, wq, np.full(K // 32, 126, np.uint8)) == 128 * 0.75 * 0.5 + 128 * 0.75 * 3.0


@pytest.fixture(scope="module")
def mx_case(oracle_mod):
    x = inputs.make_mx("tiny_mxfp4")
    ids, wts = oracle_mod.route(x.hidden, x.router_w, None, x.shape.top_k)
    out, d = oracle_mod.mxfp4_forward(x.hidden, ids, wts, x.w13, x.s13, x.w2, x.s2, debug=True)
    return x, ids, wts, out, d


def test_mx_gate_up_and_down_within_float64_bound(mx_case):
    x, ids, _, _, d = mx_case
    H, I = x.shape.hidden, x.shape.inter
    a = dec_e4m3(d["qa"]) * np.repeat(d["sa"].astype(np.float64), 128, -1)
    for t in range(x.M):
        for j in range(x.shape.top_k):
            W = deq_mx(x.w13[ids[t, j]], x.s13[ids[t, j]])      # [2I][H]
            G = W @ a[t]
            bound = (1 + 4 + 2 + H // 128 + 2) * U * (np.abs(W) @ np.abs(a[t])) * 1.01 + 1e-35
            got = np.concatenate([d["g"][t, j], d["u"][t, j]])
            assert np.all(np.abs(got - G) <= bound), (t, j)
            ac = dec_e4m3(d["qact"][t, j]) * np.repeat(d["s2"][t, j].astype(np.float64), 128)
            W2 = deq_mx(x.w2[ids[t, j]], x.s2[ids[t, j]])       # [H][I]
            Y = W2 @ ac
            bound = (1 + 4 + 2 + I // 128 + 2) * U * (np.abs(W2) @ np.abs(ac)) * 1.01 + 1e-35
            assert np.all(np.abs(d["y"][t, j] - Y) <= bound), (t, j)


def test_mx_activation_and_combine_follow_the_fp8_layer(mx_case, oracle_mod):
    x, ids, wts, out, d = mx_case
    q, s = oracle_mod.quantise(d["act"])
    assert np.array_equal(q, d["qact"]) and np.array_equal(s, d["s2"])
    # the combine: slots ascending, FP32 multiply then add, BF16
    y = d["y"]
    acc = np.zeros((x.M, x.shape.hidden), np.float32)
    for j in range(x.shape.top_k):
        acc = (acc + (wts[:, j:j + 1] * y[:, j]).astype(np.float32)).astype(np.float32)
    assert np.array_equal(oracle_mod.bf16_round(acc), out)


def test_mx_dense_brute_force_equals_sparse(mx_case, oracle_mod):
    x, ids, wts, out, _ = mx_case
    M, E, H = x.M, x.shape.num_experts, x.shape.hidden
    ydense = np.zeros((E, M, H), np.float32)
    for e in range(E):
        _, dd = oracle_mod.mxfp4_forward(x.hidden[:M], np.full((M, 1), e, np.int32), np.ones((M, 1), np.float32),
                                         x.w13, x.s13, x.w2, x.s2, debug=True)
        ydense[e] = dd["y"][:, 0]
    acc = np.zeros((M, H), np.float32)
    for j in range(x.shape.top_k):
        acc = (acc + (wts[:, j:j + 1] * ydense[ids[:, j], np.arange(M)]).astype(np.float32)).astype(np.float32)
    assert np.array_equal(oracle_mod.bf16_round(acc), out)


def test_mx_equals_fp8_layer_on_fp8_exact_weights(oracle_mod):
    """Weights whose every 32-block scale is 2^0 are E4M3-exact; with sub-block sums that
    stay exact in FP32 (small-integer data) the MXFP4 oracle equals the FP8 oracle with unit
    block scales bit for bit -- two independent loops over the same arithmetic."""
    H, I, E, K, M = 256, 128, 4, 2, 3
    g = np.random.default_rng(11)
    codes13 = g.integers(0, 16, (E, 2 * I, H)).astype(np.uint8)
    codes2 = g.integers(0, 16, (E, H, I)).astype(np.uint8)
    pack = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    to_e4m3 = lambda c: torch.from_numpy(e2m1_dec(c).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    xv = g.choice(np.array([0.0, 1.0, -1.0, 2.0, -2.0, 0.5]), (M, H)).astype(np.float32)
    xv[:, 0] = 448.0
    xv[:, 128] = 448.0  # hidden scales exactly 1
    hidden = inputs.to_bf16_bits(xv)
    ids = np.array([[0, 3], [1, 2], [2, 2]], np.int32)
    wts = np.array([[0.5, 0.5], [0.25, 0.75], [1.0, 0.0]], np.float32)
    mx = oracle_mod.mxfp4_forward(hidden, ids, wts, pack(codes13), np.full((E, 2 * I, H // 32), 127, np.uint8),
                                  pack(codes2), np.full((E, H, I // 32), 127, np.uint8))
    fp8 = oracle_mod.moe_forward(hidden, ids, wts, to_e4m3(codes13), np.ones((E, 2 * I // 128, H // 128), np.float32),
                                 to_e4m3(codes2), np.ones((E, H // 128, I // 128), np.float32))
    assert np.array_equal(mx, fp8)


def test_mx_zero_rows_and_invalid_ids(mx_case, oracle_mod):
    x, ids, wts, _, _ = mx_case
    hid = x.hidden.copy()
    hid[1] = 0
    bad = ids.copy()
    bad[2, 0] = -1
    out = oracle_mod.mxfp4_forward(hid, bad, wts, x.w13, x.s13, x.w2, x.s2)
    assert np.all(out[1] == 0)
    one = oracle_mod.mxfp4_forward(hid[2:3], ids[2:3, 1:], wts[2:3, 1:], x.w13, x.s13, x.w2, x.s2)
    assert np.array_equal(out[2], one[0])
