"""Pins for the oracle's expert FFN (gate/up block GEMM, SiLU*up requantisation, down block
GEMM) and its fixed-order combine.

Stages follow docs/compiler/architecture.md (accepted M=1 MoE objects: gate/up, SiLU+quant,
down/reduce) and the netra-kernel README prefill-pair section (a route reducer with its own
fixed reduction order); "Inferact/amd-kernels" README (partials summed in a fixed order,
never with atomics). Every pin is independent of the oracle's loops: float64 library
matmuls over torch-decoded weights with a rigorous rounding bound, scipy's expit, closed
forms, and brute force over all experts.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

from fp8_block_scaled_router_gb300 import inputs

U = 2.0 ** -24


def dec(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def deq_weight(codes, scales):
    """[N][Kd] codes, [N/128][Kd/128] scales -> float64 dequantised matrix."""
    s = np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1)
    return dec(codes) * s


def deq_act(q, s):
    return dec(q) * np.repeat(s.astype(np.float64), 128, -1)


def tiny(E=None, M=None):
    return inputs.make("tiny", E=E, M=M)


def run(oracle_mod, x, ids=None, wts=None, nthreads=1):
    if ids is None:
        ids, wts = oracle_mod.route(x.hidden, x.router_w, x.bias, x.shape.top_k)
    out, d = oracle_mod.moe_forward(x.hidden, ids, wts, x.w13, x.s13, x.w2, x.s2, debug=True,
                                    nthreads=nthreads)
    return ids, wts, out, d


CASES = [("tiny", None, None), ("decode", 16, 3), ("wide", 8, 2)]


@pytest.fixture(scope="module", params=CASES, ids=[c[0] for c in CASES])
def case(request, oracle_mod):
    name, E, M = request.param
    x = inputs.make(name, E=E, M=M)
    ids, wts, out, d = run(oracle_mod, x, nthreads=4)
    return x, ids, wts, out, d


def test_gate_up_within_float64_bound(case):
    x, ids, _, _, d = case
    H, I = x.shape.hidden, x.shape.inter
    a = deq_act(d["qa"], d["sa"])                            # [M][H]
    nkb = H // 128
    for t in range(x.M):
        for j in range(x.shape.top_k):
            W = deq_weight(x.w13[ids[t, j]], x.s13[ids[t, j]])  # [2I][H]
            G = W @ a[t]
            Gabs = np.abs(W) @ np.abs(a[t])
            bound = (nkb + 3) * U * Gabs * 1.01 + 1e-35
            got = np.concatenate([d["g"][t, j], d["u"][t, j]])
            assert np.all(np.abs(got - G) <= bound), (t, j)
            # gabs/uabs report the magnitude of the promoted partial sums
            assert np.all(np.concatenate([d["gabs"][t, j], d["uabs"][t, j]]) <= Gabs * (1 + 1e-5))


def test_silu_mul_matches_expit(case):
    _, _, _, _, d = case
    g, u = d["g"].astype(np.float64), d["u"].astype(np.float64)
    ref = g * expit(g) * u
    assert np.all(np.abs(d["act"] - ref) <= 2 * U * np.abs(ref) + 1e-38)


def test_activation_requantised_per_128(case, oracle_mod):
    x, _, _, _, d = case
    q, s = oracle_mod.quantise(d["act"])
    assert np.array_equal(q, d["qact"]) and np.array_equal(s, d["s2"])
    amax = np.abs(d["act"]).reshape(*d["act"].shape[:-1], -1, 128).max(-1)
    assert np.array_equal(d["s2"], np.where(amax > 0, (amax / np.float32(448)).astype(np.float32),
                                            np.float32(1)))


def test_hidden_quantised_per_token_per_128(case, oracle_mod):
    x, _, _, _, d = case
    q, s = oracle_mod.quantise(inputs.bf16_bits_to_f32(x.hidden[: x.M]))
    assert np.array_equal(q, d["qa"]) and np.array_equal(s, d["sa"])


def test_down_within_float64_bound(case):
    x, ids, _, _, d = case
    I = x.shape.inter
    nkb = I // 128
    for t in range(x.M):
        for j in range(x.shape.top_k):
            a = deq_act(d["qact"][t, j], d["s2"][t, j])
            W = deq_weight(x.w2[ids[t, j]], x.s2[ids[t, j]])  # [H][I]
            Y = W @ a
            bound = (nkb + 3) * U * (np.abs(W) @ np.abs(a)) * 1.01 + 1e-35
            assert np.all(np.abs(d["y"][t, j] - Y) <= bound), (t, j)


def test_combine_within_bf16_rounding(case):
    x, _, wts, out, d = case
    y = d["y"].astype(np.float64)
    ref = np.einsum("tk,tkh->th", wts.astype(np.float64), y)
    absr = np.einsum("tk,tkh->th", np.abs(wts.astype(np.float64)), np.abs(y))
    K = x.shape.top_k
    got = inputs.bf16_bits_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + (2 * K + 2) * U * absr * 1.01 + 1e-38)


def test_dense_brute_force_equals_sparse(oracle_mod):
    """Evaluate every expert for every token (one expert per call) and combine the routed
    ones by hand: bit-identical to the sparse evaluation."""
    x = tiny()
    ids, wts, out, _ = run(oracle_mod, x)
    M, E, H = x.M, x.shape.num_experts, x.shape.hidden
    ydense = np.zeros((E, M, H), np.float32)
    for e in range(E):
        _, d = oracle_mod.moe_forward(x.hidden[:M], np.full((M, 1), e, np.int32),
                                      np.ones((M, 1), np.float32), x.w13, x.s13, x.w2, x.s2,
                                      debug=True)
        ydense[e] = d["y"][:, 0]
    for t in range(M):
        acc = np.float32(0)
        accs = []
        for h in range(H):
            acc = np.float32(0)
            for j in range(x.shape.top_k):
                acc = np.float32(acc + np.float32(wts[t, j] * ydense[ids[t, j], t, h]))
            accs.append(acc)
        assert np.array_equal(oracle_mod.bf16_round(np.array(accs, np.float32)), out[t])


def test_identical_experts_ignore_ids(oracle_mod):
    x = tiny()
    E = x.shape.num_experts
    w13 = np.repeat(x.w13[:1], E, 0)
    s13 = np.repeat(x.s13[:1], E, 0)
    w2 = np.repeat(x.w2[:1], E, 0)
    s2 = np.repeat(x.s2[:1], E, 0)
    g = np.random.default_rng(5)
    wts = g.dirichlet(np.ones(2), size=x.M).astype(np.float32)
    outs = []
    for seed in range(3):
        ids = np.random.default_rng(seed).integers(0, E, (x.M, 2)).astype(np.int32)
        outs.append(oracle_mod.moe_forward(x.hidden, ids, wts, w13, s13, w2, s2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_zero_rows_give_exact_zero(oracle_mod):
    x = inputs.make("tiny", zero_rows=np.array([1, 3]))
    ids, wts, out, d = run(oracle_mod, x)
    assert np.all(out[[1, 3]] == 0) and np.any(out[0] != 0)
    assert np.all(d["qa"][[1, 3]] == 0) and np.all(d["sa"][[1, 3]] == 1.0)
    assert np.all(d["s2"][[1, 3]] == 1.0) and np.all(d["y"][[1, 3]] == 0)


def test_identity_expert_closed_form(oracle_mod):
    """gate rows = c * e_i, up rows = e_i, down rows scatter column i back: with E4M3-exact
    hidden values and a 448 anchor per 128-block (so every hidden scale is exactly 1),
    out[h] = bf16(sum_j w_j * deq(Q(silu(c x_h) x_h))[h]) for h < I and 0 elsewhere."""
    H, I, E, K, M = 256, 128, 8, 2, 3
    c = 0.5
    g = np.random.default_rng(9)
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 12.0, -0.5, -1.0, -2.0, -3.0, -8.0])
    x = g.choice(vals, (M, H)).astype(np.float32)
    x[:, 0] = 448.0
    x[:, 128] = -448.0
    hidden = inputs.to_bf16_bits(x)
    one = 0x38  # E4M3 code of 1.0
    w13 = np.zeros((E, 2 * I, H), np.uint8)
    w2 = np.zeros((E, H, I), np.uint8)
    for i in range(I):
        w13[:, i, i] = one
        w13[:, I + i, i] = one
        w2[:, i, i] = one
    s13 = np.ones((E, 2 * I // 128, H // 128), np.float32)
    s13[:, : I // 128, :] = c
    s2w = np.ones((E, H // 128, I // 128), np.float32)
    ids = np.array([[1, 6], [0, 7], [3, 3]], np.int32)
    wts = np.array([[0.75, 0.25], [0.5, 0.5], [0.625, 0.375]], np.float32)
    out = oracle_mod.moe_forward(hidden, ids, wts, w13, s13, w2, s2w)
    # closed form, with torch's float8 cast for the requantisation
    xs = x[:, :I].astype(np.float64)
    act = (c * xs / (1.0 + np.exp(-c * xs)) * xs).astype(np.float32)
    amax = np.abs(act).max(1, keepdims=True)
    s = np.where(amax > 0, amax / np.float32(448), np.float32(1)).astype(np.float32)
    q = torch.from_numpy((act / s).astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    y = (q * s).astype(np.float32)
    ref = np.zeros((M, H), np.float32)
    ref[:, :I] = (np.float32(0) + (wts[:, :1] * y).astype(np.float32)).astype(np.float32)
    ref[:, :I] = (ref[:, :I] + (wts[:, 1:] * y).astype(np.float32)).astype(np.float32)
    expect = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, expect)


def test_invalid_ids_contribute_nothing(oracle_mod):
    x = tiny()
    ids, wts = oracle_mod.route(x.hidden, x.router_w, None, 2)
    bad = ids.copy()
    bad[0, 1] = -1
    bad[2, 0] = 99
    out_bad = oracle_mod.moe_forward(x.hidden, bad, wts, x.w13, x.s13, x.w2, x.s2)
    # the same tokens with the bad slot removed (a K=1 call on the remaining slot)
    out0 = oracle_mod.moe_forward(x.hidden[:1], ids[:1, :1], wts[:1, :1], x.w13, x.s13, x.w2, x.s2)
    out2 = oracle_mod.moe_forward(x.hidden[2:3], ids[2:3, 1:], wts[2:3, 1:], x.w13, x.s13, x.w2, x.s2)
    assert np.array_equal(out_bad[0], out0[0]) and np.array_equal(out_bad[2], out2[0])


def test_threads_do_not_change_results(oracle_mod):
    x = inputs.make("verify", E=16, M=6)
    ids, wts = oracle_mod.route(x.hidden, x.router_w, x.bias, 8)
    a = oracle_mod.moe_forward(x.hidden, ids, wts, x.w13, x.s13, x.w2, x.s2, nthreads=1)
    b = oracle_mod.moe_forward(x.hidden, ids, wts, x.w13, x.s13, x.w2, x.s2, nthreads=3)
    assert np.array_equal(a, b)


def test_down_combine_from_given_codes(case, oracle_mod):
    """down_combine (steps 6-7 from given activation codes): fed the forward's own codes it
    reproduces the forward's output bitwise; fed perturbed codes, its output matches a
    float64 dequantised down projection and combine of those codes within the FP32 and
    BF16 rounding bound, and only the perturbed token's row changes."""
    x, ids, wts, out, d = case
    same = oracle_mod.down_combine(d["qact"], d["s2"], ids, wts, x.w2, x.s2, nthreads=2)
    assert np.array_equal(same, out)
    q = d["qact"].copy()
    t0 = x.M - 1
    q[t0, 0, 5] ^= 0x01                   # one activation code one step away
    q[t0, x.shape.top_k - 1, 130 % x.shape.inter] ^= 0x08
    got = oracle_mod.down_combine(q, d["s2"], ids, wts, x.w2, x.s2)
    assert np.array_equal(got[:t0], out[:t0])
    assert not np.array_equal(got[t0], out[t0])
    I = x.shape.inter
    nkb = I // 128
    K = x.shape.top_k
    for t in range(x.M):
        ref = np.zeros(x.shape.hidden)
        absr = np.zeros(x.shape.hidden)
        for j in range(K):
            a = deq_act(q[t, j], d["s2"][t, j])
            W = deq_weight(x.w2[ids[t, j]], x.s2[ids[t, j]])
            Y = W @ a
            ybound = (nkb + 3) * U * (np.abs(W) @ np.abs(a)) * 1.01
            ref += wts[t, j] * Y
            absr += abs(wts[t, j]) * (np.abs(Y) + ybound)
        g = inputs.bf16_bits_to_f32(got[t]).astype(np.float64)
        assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + (2 * K + 2) * U * absr * 1.01 +
                      (nkb + 3) * U * absr * 1.01 + 1e-38), t
