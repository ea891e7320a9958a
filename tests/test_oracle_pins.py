"""Pins of the CPU oracle to things other than itself (closed forms, brute
force, invariants, special cases that reduce to a dense MLP, the MX format
table). CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from moe_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(a):
    """Round-to-nearest-even fp32 -> bf16 bits (test helper, numpy)."""
    return synth.to_u16(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16))


def bf16(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def tiny_layer(copy=0, shape=synth.TINY):
    Wg = synth.to_u16(synth.router_weight(shape, copy))
    experts = {e: tuple(synth.to_u16(m) for m in synth.expert_weights(shape, copy, e))
               for e in range(shape.n_experts)}
    shared = tuple(synth.to_u16(m) for m in synth.shared_weights(shape, copy))
    return Wg, experts, shared


def dense_swiglu_f64(x, W1, W3, W2):
    """Textbook dense SwiGLU MLP in float64: W2 (silu(W1 x) * (W3 x))."""
    x = np.asarray(x, np.float64)
    g = bf16(W1).astype(np.float64) @ x
    u = bf16(W3).astype(np.float64) @ x
    h = g / (1.0 + np.exp(-g)) * u
    return bf16(W2).astype(np.float64) @ h


# ---------------------------------------------------------------- formats

def test_bf16_decode_closed_form(oracle):
    assert oracle.bf16_to_f32(np.array([0x3F80], np.uint16))[0] == 1.0
    assert oracle.bf16_to_f32(np.array([0xC000], np.uint16))[0] == -2.0
    assert oracle.bf16_to_f32(np.array([0x0001], np.uint16))[0] == math.ldexp(1.0, -133)
    lib = oracle._load()
    for b, v in ((0x3F80, 1.0), (0x4049, 3.140625), (0xBF00, -0.5)):
        assert lib.oracle_bf16_to_f32(b) == v


def test_mxfp4_table_matches_mx_spec(oracle):
    spec = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))["code_to_value"]
    for code in range(16):
        for s in range(255):
            want = math.ldexp(spec[str(code)], s - 127)
            got = oracle.mxfp4_value(code, s)
            with np.errstate(over="ignore"):
                assert got == np.float32(want), (code, s, got, want)
            if want == 0.0:
                assert math.copysign(1.0, got) == math.copysign(1.0, spec[str(code)])
        assert math.isnan(oracle.mxfp4_value(code, 255))


def test_mxfp4_decode_nibble_order_and_blocks(oracle):
    # element 2j sits in the low nibble of byte j; one scale per 32 elements
    spec = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))["code_to_value"]
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 256, size=(3, 32), dtype=np.uint8)   # K = 64
    scales = rng.integers(100, 140, size=(3, 2), dtype=np.uint8)
    out = oracle.mxfp4_decode(codes, scales, 64)
    for r in range(3):
        for c in range(64):
            byte = int(codes[r, c // 2])
            code = byte & 15 if c % 2 == 0 else byte >> 4
            assert out[r, c] == np.float32(math.ldexp(spec[str(code)], int(scales[r, c // 32]) - 127))


def test_quantiser_roundtrip_on_representable_values(oracle):
    spec = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))["code_to_value"]
    rng = np.random.default_rng(1)
    rows, K = 8, 128
    vals = np.zeros((rows, K), np.float32)
    for r in range(rows):
        for b in range(K // 32):
            s = int(rng.integers(90, 140))
            codes = rng.integers(0, 16, size=32)
            codes[0] = 7  # block max is 6 * 2^(s-127): the quantiser then picks scale s
            vals[r, b * 32:(b + 1) * 32] = [math.ldexp(spec[str(int(c))], s - 127) for c in codes]
    q, sc = synth.mxfp4_quantize(torch.from_numpy(vals))
    back = oracle.mxfp4_decode(q.numpy(), sc.numpy(), K)
    np.testing.assert_array_equal(back, vals)


def test_quantiser_error_bound(oracle):
    w = synth.expert_weights(synth.TINY, 0, 5)[0]
    q, sc = synth.mxfp4_quantize(w)
    back = oracle.mxfp4_decode(q.numpy(), sc.numpy(), w.shape[1])
    v = w.float().numpy()
    scale = np.repeat(np.ldexp(1.0, sc.numpy().astype(np.int32) - 127), 32, axis=1)
    # the scaled block maximum lies in [4, 8): values in (6, 8) saturate at 6
    # (error < 2 steps of 2^(E-127)); all others round to a grid of step <= 2
    # (error <= 1 step)
    err = np.abs(back - v)
    assert np.all(err <= 2.0 * scale)
    assert np.all((err <= 1.0 * scale) | (np.abs(v) > 6.0 * scale))


# ---------------------------------------------------------------- routing

def test_router_logits_match_exact_dot_within_fp32_bound(oracle):
    Wg, _, _ = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 0, 4))
    _, _, logits = oracle.route(x, Wg, 2)
    exact = bf16(x).astype(np.float64) @ bf16(Wg).astype(np.float64).T
    H = x.shape[1]
    gamma = H * 2.0 ** -24 / (1 - H * 2.0 ** -24)
    bound = gamma * (np.abs(bf16(x)).astype(np.float64) @ np.abs(bf16(Wg)).astype(np.float64).T)
    assert np.all(np.abs(logits - exact) <= bound + 1e-30)


def test_topk_brute_force_over_all_subsets(oracle):
    Wg, _, _ = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 7, 16))
    k = 2
    idx, w, logits = oracle.route(x, Wg, k)
    E = Wg.shape[0]
    for t in range(x.shape[0]):
        best = None
        for sub in itertools.combinations(range(E), k):  # lexicographic order
            s = sum(float(logits[t, e]) for e in sub)
            if best is None or s > best[0]:
                best = (s, sub)
        assert set(idx[t]) == set(best[1])
        assert logits[t, idx[t, 0]] >= logits[t, idx[t, 1]]


def test_topk_matches_stable_sort_and_ties_go_low(oracle):
    Wg, _, _ = tiny_layer()
    Wg = Wg.copy()
    Wg[9] = Wg[3]    # duplicated rows give exactly tied logits
    Wg[12] = Wg[3]
    x = synth.to_u16(synth.x_independent(synth.TINY, 11, 8))
    for k in (1, 2, 5, 16):
        idx, _, logits = oracle.route(x, Wg, k)
        for t in range(x.shape[0]):
            order = sorted(range(Wg.shape[0]), key=lambda e: (-float(logits[t, e]), e))
            assert list(idx[t]) == order[:k]


def test_weights_sum_to_one_and_special_k(oracle):
    Wg, _, _ = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 3, 6))
    idx, w, logits = oracle.route(x, Wg, 2)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-6)
    idx1, w1, _ = oracle.route(x, Wg, 1)
    assert np.all(w1 == 1.0)
    np.testing.assert_array_equal(idx1[:, 0], np.argmax(logits, axis=1))
    E = Wg.shape[0]
    idxE, wE, _ = oracle.route(x, Wg, E)
    for t in range(x.shape[0]):
        l = logits[t].astype(np.float64)
        p = np.exp(l - l.max())
        p /= p.sum()
        np.testing.assert_allclose(wE[t], p[idxE[t]], rtol=2e-6, atol=1e-9)


def test_zero_input(oracle):
    Wg, experts, shared = tiny_layer()
    x = np.zeros((3, 256), np.uint16)
    idx, w, logits = oracle.route(x, Wg, 2)
    assert np.all(logits == 0)
    assert np.all(idx == np.array([0, 1]))
    assert np.all(w == 0.5)
    y = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    assert np.all(y == 0)


# ---------------------------------------------------------------- experts and combine

def test_closed_form_hand_example(oracle):
    """E=4, k=2, H=32, I=Is=2; x = e_0 so every projection reads column 0 and
    every value below is a closed form."""
    H, I, E, k = 32, 2, 4, 2
    x = np.zeros((1, H), np.float32); x[0, 0] = 1.0
    c = [0.5, 2.0, -1.0, 1.0]                     # logits
    Wg = np.zeros((E, H), np.float32); Wg[:, 0] = c
    gate = {1: [1.0, -2.0], 3: [0.5, 3.0], "s": [-1.0, 2.0]}
    up = {1: [2.0, 0.5], 3: [-1.0, 1.0], "s": [1.0, 1.0]}
    W2map = [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [1.0, -1.0]]   # rows o = 0..3

    def mats(key):
        W1 = np.zeros((I, H), np.float32); W1[:, 0] = gate[key]
        W3 = np.zeros((I, H), np.float32); W3[:, 0] = up[key]
        W2 = np.zeros((H, I), np.float32); W2[:4] = W2map
        if key == 3:
            W2[:4] = np.array(W2map)[:, ::-1]
        return tuple(f32_to_bf16_bits(m) for m in (W1, W3, W2))

    experts = {e: mats(e if e in (1, 3) else 1) for e in range(E)}
    experts[0] = mats(1); experts[2] = mats(1)
    shared = mats("s")
    xb, Wgb = f32_to_bf16_bits(x), f32_to_bf16_bits(Wg)
    idx, w, _ = oracle.route(xb, Wgb, k)
    assert list(idx[0]) == [1, 3]
    w_want = [1.0 / (1.0 + math.exp(-1.0)), 1.0 / (1.0 + math.exp(1.0))]
    np.testing.assert_allclose(w[0], w_want, rtol=1e-6)

    def silu(v):
        return v / (1.0 + math.exp(-v))

    def z(key, flip):
        h = [silu(gate[key][i]) * up[key][i] for i in range(I)]
        rows = np.array(W2map)[:, ::-1] if flip else np.array(W2map)
        out = np.zeros(H)
        out[:4] = rows @ np.array(h)
        return out

    y_want = w_want[0] * z(1, False) + w_want[1] * z(3, True) + z("s", False)
    y = oracle.ffn(xb, idx, w, experts, E, I, shared)
    np.testing.assert_allclose(y[0], y_want, rtol=2e-6, atol=1e-7)
    yd = oracle.ffn(xb, idx, w, experts, E, I, shared, acc_double=True)
    np.testing.assert_allclose(yd[0], y_want, rtol=3e-7, atol=1e-7)  # w and z are stored as fp32


def test_identical_experts_collapse_to_dense_mlp(oracle):
    Wg, experts, shared = tiny_layer()
    same = experts[4]
    experts = {e: same for e in range(16)}
    x = synth.to_u16(synth.x_independent(synth.TINY, 5, 4))
    idx, w, _ = oracle.route(x, Wg, 2)
    y = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    for t in range(4):
        want = dense_swiglu_f64(bf16(x[t]), *same) + dense_swiglu_f64(bf16(x[t]), *shared)
        np.testing.assert_allclose(y[t], want, rtol=1e-5, atol=1e-6)


def test_single_expert_layer_reduces_to_weighted_dense_mlp(oracle):
    # distinct experts, one token: y = sum_j w_j MLP_j(x) + MLP_s(x), each
    # MLP a textbook float64 dense SwiGLU; weights from the closed-form softmax
    Wg, experts, shared = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 9, 1))
    idx, w, logits = oracle.route(x, Wg, 2)
    l = logits[0].astype(np.float64)
    p = np.exp(l[idx[0]] - l.max())
    w_want = p / p.sum()
    np.testing.assert_allclose(w[0], w_want, rtol=1e-6)
    want = sum(w_want[j] * dense_swiglu_f64(bf16(x[0]), *experts[int(idx[0, j])]) for j in range(2))
    want = want + dense_swiglu_f64(bf16(x[0]), *shared)
    y = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    np.testing.assert_allclose(y[0], want, rtol=1e-5, atol=1e-6)


def test_joint_expert_permutation_invariance(oracle):
    Wg, experts, shared = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 2, 5))
    idx, w, _ = oracle.route(x, Wg, 2)
    y = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    perm = np.random.default_rng(3).permutation(16)     # expert e -> perm[e]
    Wg_p = np.empty_like(Wg)
    Wg_p[perm] = Wg
    experts_p = {int(perm[e]): m for e, m in experts.items()}
    idx_p, w_p, _ = oracle.route(x, Wg_p, 2)
    np.testing.assert_array_equal(idx_p, perm[idx])
    # the fp32 softmax denominator sums over experts in index order, so a
    # permutation may move w by an ulp; y follows within 1e-6
    np.testing.assert_allclose(w_p, w, rtol=1e-6)
    y_p = oracle.ffn(x, idx_p, w_p, experts_p, 16, 64, shared)
    np.testing.assert_allclose(y_p, y, rtol=1e-6, atol=1e-7)
    y_same_w = oracle.ffn(x, idx_p, w, experts_p, 16, 64, shared)
    np.testing.assert_array_equal(y_same_w, y)


def test_token_independence(oracle):
    Wg, experts, shared = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 4, 6))
    idx, w, logits = oracle.route(x, Wg, 2)
    y = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    for t in range(6):
        i1, w1, l1 = oracle.route(x[t:t + 1], Wg, 2)
        np.testing.assert_array_equal(i1[0], idx[t])
        np.testing.assert_array_equal(w1[0], w[t])
        np.testing.assert_array_equal(l1[0], logits[t])
        y1 = oracle.ffn(x[t:t + 1], i1, w1, experts, 16, 64, shared)
        np.testing.assert_array_equal(y1[0], y[t])


def test_fp32_oracle_within_1e5_of_fp64(oracle):
    Wg, experts, shared = tiny_layer()
    x = synth.to_u16(synth.x_independent(synth.TINY, 1, 8))
    idx, w, _ = oracle.route(x, Wg, 2)
    y32 = oracle.ffn(x, idx, w, experts, 16, 64, shared)
    y64 = oracle.ffn(x, idx, w, experts, 16, 64, shared, acc_double=True)
    assert np.linalg.norm(y32 - y64) / np.linalg.norm(y64) < 1e-5


def test_mxfp4_expert_equals_bf16_expert_on_dequantised_weights(oracle):
    W1, W3, W2 = synth.expert_weights(synth.TINY, 0, 2)
    H, I = 256, 64
    q = [synth.mxfp4_quantize(m) for m in (W1, W3, W2)]
    deq = [oracle.mxfp4_decode(c.numpy(), s.numpy(), m.shape[1]) for (c, s), m in zip(q, (W1, W3, W2))]
    deq_bf16 = [f32_to_bf16_bits(d) for d in deq]
    for d, b in zip(deq, deq_bf16):
        np.testing.assert_array_equal(bf16(b), d)   # e2m1 x 2^k is bf16-exact
    x = bf16(synth.to_u16(synth.x_independent(synth.TINY, 0, 1))[0])
    z4 = oracle.expert(x, q[0][0].numpy(), q[1][0].numpy(), q[2][0].numpy(), wfmt=1,
                       S=(q[0][1].numpy(), q[1][1].numpy(), q[2][1].numpy()))
    zb = oracle.expert(x, *deq_bf16)
    np.testing.assert_array_equal(z4, zb)


@pytest.mark.slow_cpu
def test_ling_single_token_fp32_vs_fp64(oracle):
    shape = synth.LING
    Wg = synth.to_u16(synth.router_weight(shape, 0))
    x = synth.to_u16(synth.x_independent(shape, 0, 1))
    idx, w, _ = oracle.route(x, Wg, 8)
    idx64, w64, _ = oracle.route(x, Wg, 8, acc_double=True)
    assert set(idx[0]) == set(idx64[0])
    np.testing.assert_allclose(w, w64, rtol=1e-5)
    experts = {int(e): tuple(synth.to_u16(m) for m in synth.expert_weights(shape, 0, int(e)))
               for e in idx[0]}
    shared = tuple(synth.to_u16(m) for m in synth.shared_weights(shape, 0))
    y32 = oracle.ffn(x, idx, w, experts, 512, 768, shared)
    y64 = oracle.ffn(x, idx, w, experts, 512, 768, shared, acc_double=True)
    assert np.linalg.norm(y32 - y64) / np.linalg.norm(y64) < 1e-5


# ---------------------------------------------------------------- all-core variant

@pytest.mark.parametrize("wfmt,shared", [(0, True), (0, False), (1, True), (2, True)])
def test_parallel_ffn_is_bit_identical(oracle, wfmt, shared):
    """The threaded FFN used for the all-core CPU baseline runs the same
    expert calls and combines them in the same order: the same bits as the
    single-thread oracle, for every weight format."""
    sh = synth.LayerShape(512, 16, 3, 128, 128) if wfmt == 2 else synth.LayerShape(256, 16, 3, 64, 64)
    layer = synth.device_layer(sh, 2, wfmt=wfmt, device="cpu")
    x = synth.to_u16(synth.x_independent(sh, 3, 5))
    idx, w, _ = oracle.route(x, synth.to_u16(layer["Wg"]), sh.top_k)
    experts = {int(e): synth.host_expert(sh, layer, int(e), wfmt) for e in np.unique(idx)}
    sw = tuple(synth.to_u16(layer[n]) for n in ("ws1", "ws3", "ws2")) if shared else None
    y1 = oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, sw, wfmt=wfmt)
    for nt in (0, 2, 3):
        yp = oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, sw, wfmt=wfmt, nthreads=nt)
        assert np.array_equal(y1.view(np.uint32), yp.view(np.uint32))
    yd = oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, sw, wfmt=wfmt, acc_double=True)
    ydp = oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, sw, wfmt=wfmt, acc_double=True, nthreads=0)
    assert np.array_equal(yd.view(np.uint32), ydp.view(np.uint32))


def test_parallel_ffn_rejects_a_missing_expert(oracle):
    sh = synth.TINY
    x = synth.to_u16(synth.x_independent(sh, 4, 2))
    idx = np.array([[1, 2], [3, 4]], np.int32)
    w = np.full((2, 2), 0.5, np.float32)
    experts = {e: tuple(synth.to_u16(m) for m in synth.expert_weights(sh, 0, e)) for e in (1, 2, 3)}
    with pytest.raises(ValueError):
        oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, None, nthreads=0)
