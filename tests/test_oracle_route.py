"""Pins for the oracle's router (softmax + top-k with renormalisation).

Routing is the first stage of the routed MoE producer ("NetraRuntime/netra-kernel"
README, prefill-pair build section; BF16 routing in its capability table). The pins use
float64 library arithmetic (numpy matmul, scipy softmax, numpy lexsort) with rigorous
error bounds, plus the special cases that fix the tie rule and the renormalisation.
"""
import numpy as np
import pytest
from scipy.special import softmax

from fp8_block_scaled_router_gb300 import inputs

U = 2.0 ** -24


def f32(b):
    return inputs.bf16_bits_to_f32(b)


def rand_case(seed, M, H, E, std=0.02):
    x = inputs.hidden_states(seed, M, H)
    w = inputs.router_weights(seed, H, E, std)
    return x, w


def logit_bound(x, w):
    H = x.shape[1]
    absdot = np.abs(f32(x).astype(np.float64)) @ np.abs(f32(w).astype(np.float64))
    return (128 + H // 128 + 2) * U * absdot * 1.01 + 1e-30


@pytest.mark.parametrize("M,H,E,K", [(4, 256, 8, 2), (16, 2048, 128, 8), (6, 6144, 128, 4)])
def test_logits_within_float64_bound(oracle_mod, M, H, E, K):
    x, w = rand_case(11, M, H, E)
    _, _, logits = oracle_mod.route(x, w, None, K, want_logits=True)
    ref = f32(x).astype(np.float64) @ f32(w).astype(np.float64)
    assert np.all(np.abs(logits - ref) <= logit_bound(x, w))


@pytest.mark.parametrize("renorm", [True, False])
def test_selection_and_weights_match_library(oracle_mod, renorm):
    M, H, E, K = 32, 2048, 128, 8
    x, w = rand_case(12, M, H, E)
    bias = np.linspace(-0.5, 0.5, E).astype(np.float32)
    ids, wts, logits = oracle_mod.route(x, w, bias, K, renormalize=renorm, want_logits=True)
    for t in range(M):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))  # desc, ties -> low id
        assert ids[t].tolist() == order[:K].tolist()
        sel = logits[t, ids[t]].astype(np.float64)
        ref = softmax(sel) if renorm else softmax(logits[t].astype(np.float64))[ids[t]]
        assert np.all(np.abs(wts[t] - ref) <= 1e-6 * ref)
        assert np.all(np.diff(wts[t]) <= 0)                  # slots in descending weight
        assert len(set(ids[t].tolist())) == K and ids[t].min() >= 0 and ids[t].max() < E
    if renorm:
        assert np.all(np.abs(wts.astype(np.float64).sum(1) - 1.0) <= 1e-6)


def test_bias_is_added_to_logits(oracle_mod):
    M, H, E, K = 8, 2048, 128, 8
    x, w = rand_case(13, M, H, E)
    bias = np.zeros(E, np.float32)
    bias[[0, 1, 2, 3]] = 3.0
    _, _, l0 = oracle_mod.route(x, w, None, K, want_logits=True)
    ids, _, l1 = oracle_mod.route(x, w, bias, K, want_logits=True)
    assert np.array_equal(l1, (l0 + bias).astype(np.float32))
    hot = np.isin(ids, [0, 1, 2, 3]).sum(1)
    assert hot.mean() >= 3.5  # a +3.0 bias (over 3 logit sigmas) wins nearly every slot


def test_zero_router_ties_go_to_lowest_index(oracle_mod):
    M, H, E, K = 3, 256, 8, 2
    x = inputs.hidden_states(0, M, H)
    w = np.zeros((H, E), np.uint16)
    ids, wts = oracle_mod.route(x, w, None, K)
    assert ids.tolist() == [[0, 1]] * M
    assert np.all(wts == np.float32(0.5))
    ids8, w8 = oracle_mod.route(inputs.hidden_states(0, 2, 2048), np.zeros((2048, 128), np.uint16),
                                None, 8)
    assert ids8.tolist() == [list(range(8))] * 2 and np.all(w8 == np.float32(0.125))


def test_equal_columns_tie_break(oracle_mod):
    """Duplicated router columns give bit-equal logits; the lower expert wins the slot."""
    M, H, E = 5, 256, 8
    x, w = rand_case(14, M, H, E)
    w = w.copy()
    w[:, 5] = w[:, 2]
    w[:, 7] = w[:, 2]
    ids, _, logits = oracle_mod.route(x, w, None, E, want_logits=True)
    for t in range(M):
        pos = {e: ids[t].tolist().index(e) for e in (2, 5, 7)}
        assert pos[2] < pos[5] < pos[7]
        assert pos[5] == pos[2] + 1 and pos[7] == pos[2] + 2


def test_top1_renormalised_weight_is_one(oracle_mod):
    x, w = rand_case(15, 9, 2048, 128)
    _, wts = oracle_mod.route(x, w, None, 1)
    assert np.all(wts == 1.0)


def test_topk_equals_e_gives_full_softmax(oracle_mod):
    M, H, E = 6, 256, 8
    x, w = rand_case(16, M, H, E, std=0.2)
    ids, wts, logits = oracle_mod.route(x, w, None, E, want_logits=True)
    for t in range(M):
        full = softmax(logits[t].astype(np.float64))
        assert np.all(np.abs(wts[t] - full[ids[t]]) <= 1e-6 * full[ids[t]])
        assert sorted(ids[t].tolist()) == list(range(E))


def test_zero_hidden_row(oracle_mod):
    x = np.zeros((2, 2048), np.uint16)
    _, w = rand_case(17, 1, 2048, 128)
    ids, wts = oracle_mod.route(x, w, None, 8)
    assert ids.tolist() == [list(range(8))] * 2 and np.all(wts == np.float32(0.125))
