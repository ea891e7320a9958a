"""Pins of the oracle's router variants (sigmoid or softmax scores, a
selection bias, a routed scaling factor) against brute force, closed forms
and invariants."""
import itertools
import math

import numpy as np
import pytest

from moe_decode_gb300 import synth


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    o.build()
    return o


def _inputs(E=16, H=64, M=5, seed=3):
    Wg = synth.to_u16(synth.normal_bf16(seed, 1, 0, E * H, 0.1)).reshape(E, H)
    x = synth.to_u16(synth.normal_bf16(seed, 2, 0, M * H, 1.0)).reshape(M, H)
    bias = np.asarray(synth.normal_f32(seed, 3, 0, E, 0.05).numpy(), np.float32)
    return x, Wg, bias


def _sig(v):
    return 1.0 / (1.0 + math.exp(-v))


@pytest.mark.parametrize("scoring", [0, 1])
def test_selection_is_the_best_subset_by_biased_score(oracle, scoring):
    x, Wg, bias = _inputs()
    k = 3
    idx, w, logits = oracle.route_ex(x, Wg, k, scoring=scoring, bias=bias)
    for t in range(x.shape[0]):
        l = logits[t].astype(np.float64)
        if scoring == 1:
            s = np.array([_sig(v) for v in l])
        else:
            s = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
        key = s + bias
        best = max(itertools.combinations(range(len(l)), k), key=lambda c: sum(key[list(c)]))
        assert set(idx[t]) == set(best), t
        assert list(idx[t]) == sorted(best, key=lambda e: -key[e])
        ws = s[idx[t]] / s[idx[t]].sum()
        assert np.allclose(w[t], ws, rtol=1e-5, atol=1e-7)


def test_dominant_bias_forces_the_set_and_order_follows_scores(oracle):
    x, Wg, _ = _inputs()
    chosen = [2, 9, 13]
    bias = np.zeros(16, np.float32)
    bias[chosen] = 10.0
    idx, w, logits = oracle.route_ex(x, Wg, 3, scoring=1, bias=bias)
    for t in range(x.shape[0]):
        assert sorted(idx[t]) == chosen
        assert list(idx[t]) == sorted(chosen, key=lambda e: -logits[t, e])
        # weights: the unbiased sigmoid scores, renormalised
        s = np.array([_sig(float(logits[t, e])) for e in idx[t]])
        assert np.allclose(w[t], s / s.sum(), rtol=1e-5)


def test_sigmoid_without_bias_selects_like_softmax(oracle):
    x, Wg, _ = _inputs(seed=8)
    i0, _, l0 = oracle.route_ex(x, Wg, 4, scoring=0)
    i1, w1, _ = oracle.route_ex(x, Wg, 4, scoring=1)
    assert np.array_equal(i0, i1)
    for t in range(x.shape[0]):
        a, b = i1[t, 0], i1[t, 1]
        assert w1[t, 0] / w1[t, 1] == pytest.approx(_sig(float(l0[t, a])) / _sig(float(l0[t, b])), rel=1e-5)


def test_scaling_factor_and_bias_shift(oracle):
    x, Wg, bias = _inputs(seed=11)
    i1, w1, _ = oracle.route_ex(x, Wg, 3, scoring=1, bias=bias, routed_scale=2.5)
    assert np.allclose(w1.sum(axis=1), 2.5, rtol=1e-6)
    i2, w2, _ = oracle.route_ex(x, Wg, 3, scoring=1, bias=bias + np.float32(0.25), routed_scale=2.5)
    assert np.array_equal(i1, i2)
    assert np.allclose(w1, w2, rtol=1e-6)
    i3, w3, _ = oracle.route_ex(x, Wg, 3, scoring=1, bias=bias, routed_scale=0.0)  # <= 0 means 1
    assert np.allclose(w3.sum(axis=1), 1.0, rtol=1e-6)


def test_softmax_with_bias_keeps_softmax_weight_ratios(oracle):
    x, Wg, bias = _inputs(seed=13)
    idx, w, logits = oracle.route_ex(x, Wg, 3, scoring=0, bias=bias * 50)
    for t in range(x.shape[0]):
        a, b = idx[t, 0], idx[t, 2]
        assert w[t, 0] / w[t, 2] == pytest.approx(math.exp(float(logits[t, a]) - float(logits[t, b])), rel=1e-5)
