"""Pins of the oracle's FP8 e4m3 decode and encode, its block quantiser and
its output-layer (lm_head) definition, against the OFP8 specification's
values, closed forms and invariants."""
import json
import math
import os

import numpy as np
import pytest

from moe_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    o.build()
    return o


def test_e4m3_values_match_the_spec(oracle):
    spec = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))
    for code, v in spec["code_to_value"].items():
        got = oracle.fp8_e4m3_value(int(code, 16))
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (code, got, v)
    for code in spec["nan_codes"]:
        assert math.isnan(oracle.fp8_e4m3_value(int(code, 16)))
    pos = [oracle.fp8_e4m3_value(c) for c in range(0x7f)]
    assert max(pos) == spec["max_finite"]
    assert min(v for v in pos if v > 0) == spec["min_subnormal"]
    assert all(b > a for a, b in zip(pos, pos[1:]))              # codes ordered by value
    assert all(oracle.fp8_e4m3_value(c | 0x80) == -oracle.fp8_e4m3_value(c) for c in range(0x7f))


def test_e4m3_encode_roundtrip_ties_and_saturation(oracle):
    for c in range(256):
        if c in (0x7f, 0xff):
            continue
        assert oracle.fp8_e4m3_encode(oracle.fp8_e4m3_value(c)) == c, hex(c)
    assert oracle.fp8_e4m3_encode(1.0625) == 0x38   # midpoint of 1 and 1.125: even code
    assert oracle.fp8_e4m3_encode(1.1875) == 0x3a   # midpoint of 1.125 and 1.25: even code
    assert oracle.fp8_e4m3_encode(1.07) == 0x39
    assert oracle.fp8_e4m3_encode(449.0) == 0x7e
    assert oracle.fp8_e4m3_encode(1e9) == 0x7e
    assert oracle.fp8_e4m3_encode(-1e9) == 0xfe
    assert oracle.fp8_e4m3_encode(float("nan")) == 0x7f
    assert oracle.fp8_e4m3_encode(0.0009765625) == 0x00  # half the smallest subnormal: even (zero)


def test_fp8_quantizer_error_bound_and_amax(oracle):
    w = synth.to_u16(synth.normal_bf16(7, 1, 0, 8 * 256, 0.02))
    w = w.reshape(8, 256)
    for block in (128, 256):
        codes, scales = oracle.fp8_quantize(w, block)
        wf = oracle.bf16_to_f32(w).astype(np.float64)
        for r in range(8):
            for b in range(256 // block):
                sl = slice(b * block, (b + 1) * block)
                sc = float(scales[r, b])
                amax = np.abs(wf[r, sl]).max()
                assert sc == np.float32(np.float32(amax) / np.float32(448.0))
                deq = np.array([oracle.fp8_e4m3_value(c) for c in codes[r, sl]])
                # the quotient is taken in fp32, then rounded to e4m3
                q = (wf[r, sl].astype(np.float32) / np.float32(sc)).astype(np.float64)
                # one e4m3 step around |q|: 2^(e-3) for normals, 2^-9 below 2^-6
                step = np.where(np.abs(q) >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 1e-30))) - 3), 2.0 ** -9)
                assert np.all(np.abs(deq - q) <= step / 2), (r, b)
                deq = deq * sc
                assert np.abs(deq).max() == pytest.approx(448.0 * sc, rel=1e-6)


def _tiny_lm():
    V, H = 48, 64
    W = synth.to_u16(synth.normal_bf16(11, 2, 0, V * H, 0.02)).reshape(V, H)
    x = synth.to_u16(synth.normal_bf16(12, 3, 0, 3 * H, 1.0)).reshape(3, H)
    return V, H, W, x


def test_lm_head_one_hot_selects_a_column(oracle):
    V, H, W, _ = _tiny_lm()
    one = np.zeros((1, H), np.uint16)
    one[0, 5] = 0x3F80  # 1.0
    got = oracle.lm_head(one, W, V)
    assert np.array_equal(got[0], oracle.bf16_to_f32(W[:, 5]))
    codes, scales = oracle.fp8_quantize(W, H)
    got8 = oracle.lm_head(one, codes, V, wfmt=2, scale=scales[:, 0], acc_double=True)
    want = np.array([oracle.fp8_e4m3_value(c) for c in codes[:, 5]]) * scales[:, 0].astype(np.float64)
    assert np.array_equal(got8[0], want.astype(np.float32))


def test_lm_head_linearity_permutation_and_precision(oracle):
    V, H, W, x = _tiny_lm()
    base = oracle.lm_head(x, W, V)
    x2 = (x.astype(np.uint32) + (1 << 7)).astype(np.uint16)  # exponent + 1: x * 2 (no zeros in x)
    assert np.all((x & 0x7F80) != 0)
    assert np.array_equal(oracle.lm_head(x2, W, V), 2 * base)
    perm = np.random.default_rng(0).permutation(V)
    assert np.array_equal(oracle.lm_head(x, W[perm], V), base[:, perm])
    d = oracle.lm_head(x, W, V, acc_double=True).astype(np.float64)
    assert np.linalg.norm(base - d) / np.linalg.norm(d) < 1e-6


def test_fp8_expert_equals_bf16_expert_on_exact_weights(oracle):
    """An FP8 expert whose dequantised weights are exactly bf16 values
    (e4m3 codes times power-of-two block scales) equals the bf16 expert on
    those values bit for bit: pins the e4m3 decode and the per-128 scale
    indexing of the expert path."""
    rng = np.random.default_rng(5)
    H, I = 256, 128
    def make(rows, K):
        codes = rng.integers(0, 256, (rows, K)).astype(np.uint8)
        codes[(codes & 0x7f) == 0x7f] = 0x3c              # no NaN codes
        sc = (2.0 ** rng.integers(-12, -4, (rows, K // 128))).astype(np.float32)
        val = np.array([[oracle.fp8_e4m3_value(c) for c in row] for row in codes]) * np.repeat(sc, 128, axis=1)
        bits = val.astype(np.float32).view(np.uint32)
        assert np.all((bits & 0xFFFF) == 0)               # exactly bf16
        return codes, sc, (bits >> 16).astype(np.uint16)
    c1, s1, b1 = make(I, H)
    c3, s3, b3 = make(I, H)
    c2, s2, b2 = make(H, I)
    x = oracle.bf16_to_f32(synth.to_u16(synth.normal_bf16(9, 9, 0, H, 1.0)))
    z8 = oracle.expert(x, c1, c3, c2, wfmt=2, S=(s1, s3, s2))
    zb = oracle.expert(x, b1, b3, b2, wfmt=0)
    assert np.array_equal(z8, zb)
