"""Pins of the oracle's pre-MoE RMSNorm: closed forms, scale invariance and
the bf16 rounding rule."""
import numpy as np
import pytest

from moe_decode_gb300 import synth


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    o.build()
    return o


def test_constant_row_normalises_to_gamma(oracle):
    H = 64
    h = np.full((2, H), 0x4040, np.uint16)         # 3.0
    h[1] = 0xC040                                   # -3.0
    gamma = synth.to_u16(synth.normal_bf16(3, 3, 0, H, 1.0))
    x = oracle.rmsnorm(h, gamma, 0.0)
    assert np.array_equal(x[0], gamma)              # 3 / sqrt(9) * g = g exactly
    assert np.array_equal(x[1], gamma ^ 0x8000)      # the sign flips


def test_scale_invariance_and_eps(oracle):
    H = 128
    h = synth.to_u16(synth.normal_bf16(4, 4, 0, 3 * H, 1.0)).reshape(3, H)
    gamma = synth.to_u16(synth.normal_bf16(5, 5, 0, H, 1.0))
    h4 = (h.astype(np.uint32) + (2 << 7)).astype(np.uint16)   # exponent + 2: h * 4
    assert np.all((h & 0x7F80) != 0)
    assert np.array_equal(oracle.rmsnorm(h, gamma, 0.0), oracle.rmsnorm(h4, gamma, 0.0))
    # a large eps shrinks every element towards zero
    big = oracle.bf16_to_f32(oracle.rmsnorm(h, gamma, 1e6))
    assert np.all(np.abs(big) < np.abs(oracle.bf16_to_f32(oracle.rmsnorm(h, gamma, 0.0))) + 1e-30)


def test_rounding_to_bf16_is_nearest_even(oracle):
    # one element of 1.0 and the rest chosen so that rms = 1 exactly: x = g
    H = 4
    h = np.array([[0x3F80, 0x3F80, 0x3F80, 0x3F80]], np.uint16)      # all 1.0: rms 1
    # gamma values whose product with 1 is exact; rounding only on g itself
    gamma = np.array([0x3F81, 0x3F80, 0xBF82, 0x0001], np.uint16)
    assert np.array_equal(oracle.rmsnorm(h, gamma, 0.0)[0], gamma)


def test_matches_an_independent_float64_computation(oracle):
    M, H = 4, 512
    h = synth.to_u16(synth.normal_bf16(6, 6, 0, M * H, 1.0)).reshape(M, H)
    gamma = synth.to_u16(synth.normal_bf16(7, 7, 0, H, 1.0))
    hf = oracle.bf16_to_f32(h).astype(np.float64)
    gf = oracle.bf16_to_f32(gamma).astype(np.float64)
    v = hf / np.sqrt((hf * hf).mean(axis=1, keepdims=True) + 1e-6) * gf
    b = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    want = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(oracle.rmsnorm(h, gamma, 1e-6), want)
