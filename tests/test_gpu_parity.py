"""GPU parity: the CUDA path, called through the C ABI, against the CPU
oracle on the same seeded inputs. Covers the five workloads (tiny M=1;
Ling-shape M=1, M=6 independent tokens, M=10 with ~50% consecutive overlap
plus an M = 1..16 sweep; MXFP4 experts at M=1 and M=6), uneven grids,
edge cases, determinism, PDL on/off, device-side error reporting."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from moe_decode_gb300 import build
    build.build()
    from moe_decode_gb300 import api as a
    oracle.build()
    a.set_option(a.OPT_GRID_CTAS, 0)
    a.set_option(a.OPT_WAIT_TIMEOUT_NS, 1_000_000_000)
    return a


@pytest.fixture(scope="module")
def tiny(api):
    return synth.device_layer(synth.TINY, 0)


@pytest.fixture(scope="module")
def ling(api):
    d = synth.device_layer(synth.LING, 0)
    yield d
    del d
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def ling_mxfp4(api):
    d = synth.device_layer(synth.LING, 0, wfmt=1)
    yield d
    del d
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ tiny

def test_tiny_m1(tiny):
    x = synth.x_independent(synth.TINY, 0, 1, device="cuda")
    err, _, _ = pu.compare_layer(synth.TINY, tiny, x, 0)
    assert err < 1e-2


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_tiny_m_sweep(tiny, M):
    x = synth.x_independent(synth.TINY, 100 + M, M, device="cuda")
    pu.compare_layer(synth.TINY, tiny, x, 0)


@pytest.mark.parametrize("G", [1, 3, 7, 19])
def test_tiny_uneven_grids(api, tiny, G):
    api.set_option(api.OPT_GRID_CTAS, G)
    try:
        for M in (1, 5, 16):
            x = synth.x_independent(synth.TINY, 300 + M, M, device="cuda")
            pu.compare_layer(synth.TINY, tiny, x, 0)
    finally:
        api.set_option(api.OPT_GRID_CTAS, 0)


@pytest.mark.parametrize("shape", [
    synth.LayerShape(256, 16, 16, 64, 64),    # k = E: weights are the full softmax
    synth.LayerShape(256, 16, 1, 64, 64),     # k = 1
    synth.LayerShape(256, 16, 2, 64, 0),      # no shared expert
    synth.LayerShape(512, 40, 3, 128, 192),   # Is != I, E not a multiple of 32
    synth.LayerShape(768, 1024, 16, 64, 64),  # largest E and k
])
def test_tiny_shape_variants(api, shape):
    layer = synth.device_layer(shape, 1)
    for M in (1, 7, 16):
        x = synth.x_independent(shape, 500 + M, M, device="cuda")
        pu.compare_layer(shape, layer, x, 0)


def test_zero_input(tiny):
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    idx, w, y, st = pu.run_layer(synth.TINY, tiny, x, 0)
    assert st == 0
    assert np.all(idx == np.array([0, 1]))
    assert np.all(w == 0.5)
    assert torch.count_nonzero(y.float()).item() == 0


def test_identical_tokens_share_experts(tiny):
    x = synth.x_independent(synth.TINY, 7, 1, device="cuda").repeat(16, 1)
    err, idx, _ = pu.compare_layer(synth.TINY, tiny, x, 0)
    assert all(set(r) == set(idx[0]) for r in idx)
    _, _, y, _ = pu.run_layer(synth.TINY, tiny, x, 0)
    assert torch.equal(y, y[0:1].expand_as(y))


# ------------------------------------------------------------------ Ling-shape, bf16

def test_ling_m1(ling):
    x = synth.x_independent(synth.LING, 0, 1, device="cuda")
    pu.compare_layer(synth.LING, ling, x, 0)


def test_ling_m6_independent(ling):
    for step in range(3):
        x = synth.x_independent(synth.LING, step, 6, device="cuda")
        _, idx, _ = pu.compare_layer(synth.LING, ling, x, 0)
        assert len(np.unique(idx)) >= 30  # independent tokens touch many experts


def test_ling_m10_overlap(ling):
    x = synth.x_overlap(synth.LING, 0, 10, device="cuda")
    _, idx, _ = pu.compare_layer(synth.LING, ling, x, 0)
    ov = np.mean([len(set(idx[t]) & set(idx[t - 1])) for t in range(1, 10)])
    assert 2.0 <= ov <= 6.0


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 11, 12, 13, 14, 15, 16])
def test_ling_m_sweep(ling, M):
    x = synth.x_overlap(synth.LING, 40 + M, M, device="cuda")
    pu.compare_layer(synth.LING, ling, x, 0)


def test_ling_uneven_grid(api, ling):
    api.set_option(api.OPT_GRID_CTAS, 101)
    try:
        x = synth.x_independent(synth.LING, 9, 6, device="cuda")
        pu.compare_layer(synth.LING, ling, x, 0)
    finally:
        api.set_option(api.OPT_GRID_CTAS, 0)


def test_ling_one_token_any_grid_bit_equal(api, ling):
    """One-token bf16 layers hand the activations to the down projection as
    tagged words copied along with each down chunk, with no grid barrier;
    a copy made before every CTA had stored its pair is read again. On one
    CTA the producer copies the first down chunks while the last gate/up rows
    are still being computed, so that path runs. Every row's dot products and
    the combine order do not depend on the grid: the output is the same bits
    on every grid, and matches the oracle."""
    x = synth.x_independent(synth.LING, 12, 1, device="cuda")
    ref = None
    for G in (0, 1, 19, 101):
        api.set_option(api.OPT_GRID_CTAS, G)
        try:
            idx, w, y, st = pu.run_layer(synth.LING, ling, x, 0)
        finally:
            api.set_option(api.OPT_GRID_CTAS, 0)
        assert st == 0, (G, st)
        if ref is None:
            ref = (idx, w, y)
            pu.check_layer_output(synth.LING, ling, x, idx, w, y, 0)
        else:
            assert np.array_equal(idx, ref[0]) and np.array_equal(w, ref[1]), G
            assert torch.equal(y, ref[2]), G


def test_ling_deterministic_and_pdl_bit_equal(api, ling):
    x = synth.x_independent(synth.LING, 3, 6, device="cuda")
    _, _, y1, _ = pu.run_layer(synth.LING, ling, x, 0)
    _, _, y2, _ = pu.run_layer(synth.LING, ling, x, 0)
    _, _, y3, _ = pu.run_layer(synth.LING, ling, x, 0, flags=api.F_NO_PDL)
    assert torch.equal(y1, y2)
    assert torch.equal(y1, y3)


# ------------------------------------------------------------------ MXFP4

@pytest.mark.parametrize("M", [1, 6])
def test_ling_mxfp4(ling_mxfp4, M):
    x = synth.x_independent(synth.LING, 20 + M, M, device="cuda")
    pu.compare_layer(synth.LING, ling_mxfp4, x, 1)


# ------------------------------------------------------------------ FP8

TINY_FP8 = synth.LayerShape(hidden=512, n_experts=16, top_k=2, inter=128, shared_inter=64)


@pytest.fixture(scope="module")
def ling_fp8(api):
    d = synth.device_layer(synth.LING, 0, wfmt=2)
    yield d
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [1, 6])
def test_ling_fp8(ling_fp8, M):
    x = synth.x_independent(synth.LING, 30 + M, M, device="cuda")
    pu.compare_layer(synth.LING, ling_fp8, x, 2)


@pytest.mark.parametrize("M", [1, 2, 5, 16])
def test_tiny_fp8_m_sweep(api, M):
    layer = synth.device_layer(TINY_FP8, 1, wfmt=2)
    x = synth.x_independent(TINY_FP8, 40 + M, M, device="cuda")
    pu.compare_layer(TINY_FP8, layer, x, 2)


@pytest.mark.parametrize("G", [1, 7, 19])
def test_tiny_fp8_uneven_grids(api, G):
    layer = synth.device_layer(TINY_FP8, 2, wfmt=2)
    x = synth.x_independent(TINY_FP8, 50 + G, 3, device="cuda")
    api.set_option(api.OPT_GRID_CTAS, G)
    try:
        pu.compare_layer(TINY_FP8, layer, x, 2)
    finally:
        api.set_option(api.OPT_GRID_CTAS, 0)


def test_fp8_no_shared_expert(api):
    sh = synth.LayerShape(hidden=512, n_experts=16, top_k=3, inter=256, shared_inter=0)
    layer = synth.device_layer(sh, 3, wfmt=2)
    x = synth.x_independent(sh, 60, 4, device="cuda")
    pu.compare_layer(sh, layer, x, 2)


def test_mxfp4_dequant_bit_exact(api):
    # every (code, scale) pair: row s holds codes 0..15 twice under scale s
    lo = np.arange(0, 16, 2, dtype=np.uint8)
    hi = np.arange(1, 16, 2, dtype=np.uint8)
    row = np.tile(lo | (hi << 4), 2)                       # 16 bytes = 32 codes
    codes = np.tile(row, (256, 1))
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    want = oracle.mxfp4_decode(codes, scales, 32)
    out = torch.empty((256, 32), dtype=torch.float32, device="cuda")
    api.mxfp4_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), 32, out)
    got = out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ------------------------------------------------------------------ route / ffn entry points

def test_route_only(api, ling):
    s = api.make_shape(2560, 512, 8, 768, 768, 0)
    for M in (1, 6, 16):
        x = synth.x_independent(synth.LING, 60 + M, M, device="cuda")
        ws = api.workspace(s, M)
        idx = torch.empty((M, 8), dtype=torch.int32, device="cuda")
        w = torch.empty((M, 8), dtype=torch.float32, device="cuda")
        api.route(x, ling["Wg"], s, idx, w, ws)
        assert api.read_status(ws) == 0
        idx_o, w_o, logits_o = oracle.route(synth.to_u16(x), synth.to_u16(ling["Wg"]), 8)
        pu.check_routing(idx.cpu().numpy(), w.cpu().numpy(), idx_o, w_o, logits_o, 8)


def test_ffn_given_routing_with_duplicates_and_bad_index(api, tiny):
    shape = synth.TINY
    s = api.make_shape(256, 16, 2, 64, 64, 0)
    M = 5
    x = synth.x_independent(shape, 77, M, device="cuda")
    idx = np.array([[3, 3], [0, 15], [7, 2], [5, 99], [-1, 4]], dtype=np.int32)  # dup, bad ids
    w = np.array([[0.25, 0.75], [0.5, 0.5], [0.9, 0.1], [0.6, 0.4], [0.3, 0.7]], dtype=np.float32)
    ws = api.workspace(s, M)
    y = torch.zeros((M, 256), dtype=torch.bfloat16, device="cuda")
    api.ffn(x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), pu.expert_weights_of(tiny, 0), s, y, ws)
    assert api.read_status(ws) == api.EDEVICE_BAD_INDEX
    # oracle with the invalid entries' weights zeroed (they are skipped)
    keep = (idx >= 0) & (idx < 16)
    idx_o = np.where(keep, idx, 0).astype(np.int32)
    w_o = np.where(keep, w, 0.0).astype(np.float32)
    experts = {int(e): synth.host_expert(shape, tiny, int(e)) for e in np.unique(idx_o)}
    shared = tuple(synth.to_u16(tiny[n]) for n in ("ws1", "ws3", "ws2"))
    y_o = oracle.ffn(synth.to_u16(x), idx_o, w_o, experts, 16, 64, shared)
    assert pu.rel_l2(pu.bf16_bits_to_f32(y), y_o) <= 1e-2


@pytest.mark.parametrize("seed", [5, 91])
def test_ffn_matches_layer_one_token(api, ling, seed):
    """One token: the layer runs the one-token kernel (plan built one top-k
    round at a time, CUDA-core dots); moe_ffn on the same routing runs the
    general kernel (tensor-core dots for bf16 experts). Both match the
    oracle, and each other to within the accumulation-order difference."""
    s = api.make_shape(2560, 512, 8, 768, 768, 0)
    x = synth.x_independent(synth.LING, seed, 1, device="cuda")
    idx, w, y_layer, st = pu.run_layer(synth.LING, ling, x, 0)
    assert st == 0
    assert len(set(idx[0].tolist())) == 8
    ws = api.workspace(s, 1)
    y = torch.zeros((1, 2560), dtype=torch.bfloat16, device="cuda")
    api.ffn(x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), pu.expert_weights_of(ling, 0), s, y, ws)
    assert api.read_status(ws) == 0
    experts = {int(e): synth.host_expert(synth.LING, ling, int(e)) for e in np.unique(idx)}
    shared = tuple(synth.to_u16(ling[n]) for n in ("ws1", "ws3", "ws2"))
    y_o = oracle.ffn(synth.to_u16(x), idx, w, experts, 512, 768, shared)
    f, fl = pu.bf16_bits_to_f32(y), pu.bf16_bits_to_f32(y_layer)
    assert pu.rel_l2(f, y_o) <= 1e-2 and pu.rel_l2(fl, y_o) <= 1e-2
    assert pu.rel_l2(f, fl) < 5e-3


def test_ffn_matches_layer(api, ling):
    s = api.make_shape(2560, 512, 8, 768, 768, 0)
    M = 6
    x = synth.x_independent(synth.LING, 88, M, device="cuda")
    idx, w, y_layer, st = pu.run_layer(synth.LING, ling, x, 0)
    assert st == 0
    ws = api.workspace(s, M)
    y = torch.zeros((M, 2560), dtype=torch.bfloat16, device="cuda")
    api.ffn(x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), pu.expert_weights_of(ling, 0), s, y, ws)
    assert api.read_status(ws) == 0
    assert torch.equal(y, y_layer)


# ------------------------------------------------------------------ router variants

def _router(shape, kind, seed):
    bias = synth.normal_f32(seed, 7, 0, shape.n_experts, 0.02, "cuda")
    return {"sigmoid_bias_scale": dict(scoring=1, bias=bias, scale=2.5),
            "sigmoid": dict(scoring=1, bias=None, scale=0.0),
            "softmax_bias": dict(scoring=0, bias=bias * 5, scale=0.0)}[kind]


@pytest.mark.parametrize("kind", ["sigmoid_bias_scale", "sigmoid", "softmax_bias"])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_tiny_router_variants(tiny, kind, M):
    x = synth.x_independent(synth.TINY, 70 + M, M, device="cuda")
    pu.compare_layer(synth.TINY, tiny, x, 0, router=_router(synth.TINY, kind, 80 + M))


@pytest.mark.parametrize("M", [1, 6])
def test_ling_sigmoid_bias_router(ling, M):
    x = synth.x_independent(synth.LING, 90 + M, M, device="cuda")
    pu.compare_layer(synth.LING, ling, x, 0, router=_router(synth.LING, "sigmoid_bias_scale", 95 + M))


def test_route_only_with_sigmoid_bias(api, ling):
    M = 4
    r = _router(synth.LING, "sigmoid_bias_scale", 99)
    s = pu.api_shape(synth.LING, 0, r)
    x = synth.x_independent(synth.LING, 98, M, device="cuda")
    ws = api.workspace(s, M)
    idx = torch.full((M, 8), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((M, 8), dtype=torch.float32, device="cuda")
    api.route(x, ling["Wg"], s, idx, w, ws)
    assert api.read_status(ws) == 0
    idx_o, w_o, l_o = oracle.route_ex(synth.to_u16(x), synth.to_u16(ling["Wg"]), 8, scoring=1,
                                      bias=r["bias"].cpu().numpy(), routed_scale=2.5)
    pu.check_routing(idx.cpu().numpy(), w.cpu().numpy(), idx_o, w_o, pu.ranking_keys(l_o, r), 8)
    assert np.allclose(w.cpu().numpy().sum(axis=1), 2.5, rtol=1e-5)


# ------------------------------------------------------------------ fused norm and residual

def _io(shape, seed, norm=True, residual=True, eps=1e-6):
    g = synth.normal_bf16(seed, 8, 0, shape.hidden, 1.0, "cuda") if norm else None
    return dict(gamma=g, eps=eps, residual=residual)


@pytest.mark.parametrize("norm,residual", [(True, True), (True, False), (False, True)])
@pytest.mark.parametrize("M", [1, 7])
def test_tiny_norm_and_residual(tiny, norm, residual, M):
    h = synth.normal_bf16(110 + M, 9, 0, M * synth.TINY.hidden, 3.0, "cuda").view(M, synth.TINY.hidden)
    pu.compare_layer(synth.TINY, tiny, h, 0, io=_io(synth.TINY, 120 + M, norm, residual))


@pytest.mark.parametrize("M", [1, 6])
def test_ling_norm_residual(ling, M):
    h = synth.normal_bf16(130 + M, 9, 0, M * 2560, 3.0, "cuda").view(M, 2560)
    pu.compare_layer(synth.LING, ling, h, 0, io=_io(synth.LING, 140 + M))


def test_mxfp4_norm_residual(ling_mxfp4):
    h = synth.normal_bf16(150, 9, 0, 3 * 2560, 3.0, "cuda").view(3, 2560)
    pu.compare_layer(synth.LING, ling_mxfp4, h, 1, io=_io(synth.LING, 151))


def test_residual_with_zero_experts_returns_the_input(api):
    """All expert weights zero: y = h exactly (the residual passes through
    one fp32 add of zero and one bf16 rounding)."""
    sh = synth.TINY
    layer = synth.device_layer(sh, 5)
    for n in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
        layer[n].zero_()
    h = synth.normal_bf16(160, 9, 0, 4 * sh.hidden, 3.0, "cuda").view(4, sh.hidden)
    _, _, y, st = pu.run_layer(sh, layer, h, 0, io=_io(sh, 161, norm=True, residual=True))
    assert st == 0
    assert torch.equal(y, h)


# ------------------------------------------------------------------ device failure reporting

def test_bounded_wait_reports_timeout_and_recovers(api, tiny):
    x = synth.x_independent(synth.TINY, 5, 2, device="cuda")
    s = api.make_shape(256, 16, 2, 64, 64, 0)
    ws = api.workspace(s, 2)
    y = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    api.set_option(api.OPT_WAIT_TIMEOUT_NS, 2_000_000)
    try:
        api.decode_layer(x, tiny["Wg"], pu.expert_weights_of(tiny, 0), s, y, ws,
                         flags=api.F_DEBUG_FORCE_TIMEOUT)
        assert api.read_status(ws) == api.ETIMEOUT
    finally:
        api.set_option(api.OPT_WAIT_TIMEOUT_NS, 1_000_000_000)
    api.workspace_init(ws)
    api.decode_layer(x, tiny["Wg"], pu.expert_weights_of(tiny, 0), s, y, ws)
    assert api.read_status(ws) == 0
    _, _, _, y_o = pu.oracle_layer(synth.TINY, tiny, synth.to_u16(x), 0)
    assert pu.rel_l2(pu.bf16_bits_to_f32(y), y_o) <= 1e-2


# ------------------------------------------------------------------ host buffers

def test_tokens_and_output_in_pinned_host_memory(api, ling):
    """x read from and y written to pinned host memory by the kernel itself
    (coherent CPU-GPU link): bit-equal to the device-buffer call."""
    M = 3
    x = synth.x_independent(synth.LING, 170, M, device="cuda")
    _, _, y_dev, st = pu.run_layer(synth.LING, ling, x, 0)
    assert st == 0
    s = pu.api_shape(synth.LING, 0)
    ws = api.workspace(s, M)
    xh = x.cpu().pin_memory()
    yh = torch.zeros((M, 2560), dtype=torch.bfloat16).pin_memory()
    api.decode_layer(xh, ling["Wg"], pu.expert_weights_of(ling, 0), s, yh, ws)
    assert api.read_status(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(yh, y_dev.cpu())
