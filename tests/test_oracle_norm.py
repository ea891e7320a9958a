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
    # nearest bf16 of each float64 value, found from its two bf16 neighbours
    # (no intermediate float32 rounding): the neighbour below in magnitude is
    # the float64 value truncated to 8 significant bits
    a = np.abs(v)
    e = np.floor(np.log2(a))
    ulp = np.exp2(e - 7)
    lo = np.floor(a / ulp) * ulp
    hi = lo + ulp
    lo_bits = oracle_bits(lo)
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & ((lo_bits & 1) == 1))
    mag = np.where(pick_hi, oracle_bits(hi), lo_bits)
    want = (mag | np.where(v < 0, 0x8000, 0)).astype(np.uint16)
    assert np.array_equal(oracle.rmsnorm(h, gamma, 1e-6), want)


def oracle_bits(a):
    """bf16 bit patterns of float64 values that are exactly bf16 values."""
    f = np.asarray(a, np.float64).astype(np.float32)
    assert np.array_equal(f.astype(np.float64), np.asarray(a, np.float64))
    return (f.view(np.uint32) >> 16).astype(np.uint32)


def test_rounding_ties_go_to_even_both_ways(oracle):
    """Hand-built exact ties. h = (3, 3, 3, 1, 1, 1, 1, 1) has mean square 4,
    so 1 / rms = 0.5 exactly and x_i = h_i * 0.5 * g_i without rounding
    before the final cast. With g = 1 + 2^-7, x_0 = 1.51171875 lies exactly
    halfway between the bf16 neighbours 1.5078125 (odd mantissa 65) and
    1.515625 (even, 66): nearest-even rounds up. With g = 1 + 3 * 2^-7,
    x_1 = 1.53515625 lies halfway between 1.53125 (even, 68) and 1.5390625
    (odd, 69): nearest-even rounds down, where rounding half up would not.
    x_2 is the negative of x_0's tie. The rest are exact (0.5)."""
    h = np.array([[0x4040, 0x4040, 0x4040, 0x3F80, 0x3F80, 0x3F80, 0x3F80, 0x3F80]], np.uint16)
    gamma = np.array([0x3F81, 0x3F83, 0xBF81, 0x3F80, 0x3F80, 0x3F80, 0x3F80, 0x3F80], np.uint16)
    want = np.array([0x3FC2, 0x3FC4, 0xBFC2, 0x3F00, 0x3F00, 0x3F00, 0x3F00, 0x3F00], np.uint16)
    got = oracle.rmsnorm(h, gamma, 0.0)[0]
    assert np.array_equal(got, want), [hex(v) for v in got]
    # the same values just off the tie round to the nearer neighbour
    assert oracle.bf16_to_f32(want[:2]).tolist() == [1.515625, 1.53125]
