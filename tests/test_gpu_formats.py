"""GPU parity of the MXFP4 and FP8 routed-expert paths beyond the two Ling
workloads: a small MXFP4 shape over M = 1..16 and on uneven grids, the Ling
MXFP4 layer at M = 10 and 16 (whose shared-memory carve-up differs from
M = 1 and 6), moe_route and moe_ffn with each weight format, and MXFP4
experts whose e8m0 block scales sit at the ends of the range (0, 1, 2 and
253, 254), run through the fused layer, not only the stand-alone decode."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu

# MXFP4 and FP8 need H a multiple of 512; I a multiple of 128 covers both
SMALL = synth.LayerShape(hidden=512, n_experts=16, top_k=2, inter=128, shared_inter=64)


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
def small_mx(api):
    return synth.device_layer(SMALL, 4, wfmt=1)


@pytest.mark.parametrize("M", list(range(1, 17)))
def test_small_mxfp4_m_sweep(small_mx, M):
    x = synth.x_independent(SMALL, 200 + M, M, device="cuda")
    pu.compare_layer(SMALL, small_mx, x, 1)


@pytest.mark.parametrize("G", [1, 7, 19])
def test_small_mxfp4_uneven_grids(api, small_mx, G):
    api.set_option(api.OPT_GRID_CTAS, G)
    try:
        for M in (1, 5, 16):
            x = synth.x_overlap(SMALL, 220 + M, M, device="cuda")
            pu.compare_layer(SMALL, small_mx, x, 1)
    finally:
        api.set_option(api.OPT_GRID_CTAS, 0)


@pytest.fixture(scope="module")
def ling_mx(api):
    d = synth.device_layer(synth.LING, 1, wfmt=1)
    yield d
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [10, 16])
def test_ling_mxfp4_large_m(ling_mx, M):
    x = synth.x_overlap(synth.LING, 240 + M, M, device="cuda")
    pu.compare_layer(synth.LING, ling_mx, x, 1)


# ------------------------------------------------------------------ route / ffn per format

@pytest.mark.parametrize("wfmt", [1, 2])
@pytest.mark.parametrize("M", [1, 6, 16])
def test_route_and_ffn_per_format(api, wfmt, M):
    """moe_route launches the format's kernel instantiation in route mode
    (MXFP4 layers hold the tokens in f16 times a power of two), moe_ffn its
    FFN mode; both against the oracle, and moe_ffn on the layer's own routing
    bit-equal to the fused layer."""
    layer = synth.device_layer(SMALL, 5, wfmt=wfmt)
    s = pu.api_shape(SMALL, wfmt)
    k = SMALL.top_k
    x = synth.x_independent(SMALL, 260 + M, M, device="cuda")
    ws = api.workspace(s, M)
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((M, k), dtype=torch.float32, device="cuda")
    api.route(x, layer["Wg"], s, idx, w, ws)
    assert api.read_status(ws) == 0
    idx_o, w_o, logits_o = oracle.route(synth.to_u16(x), synth.to_u16(layer["Wg"]), k)
    pu.check_routing(idx.cpu().numpy(), w.cpu().numpy(), idx_o, w_o, logits_o, k)

    y = torch.zeros((M, SMALL.hidden), dtype=torch.bfloat16, device="cuda")
    api.ffn(x, idx, w, pu.expert_weights_of(layer, wfmt), s, y, ws)
    assert api.read_status(ws) == 0
    idx_h, w_h = idx.cpu().numpy(), w.cpu().numpy()
    experts = {int(e): synth.host_expert(SMALL, layer, int(e), wfmt) for e in np.unique(idx_h)}
    shared = tuple(synth.to_u16(layer[n]) for n in ("ws1", "ws3", "ws2"))
    y_o = oracle.ffn(synth.to_u16(x), idx_h, w_h, experts, SMALL.n_experts, SMALL.inter, shared, wfmt=wfmt)
    y_g = pu.bf16_bits_to_f32(y)
    assert pu.rel_l2(y_g, y_o) <= pu.TOL_Y[wfmt]
    pu.check_per_token(y_g, y_o, pu.TOL_Y[wfmt])

    idx_l, _, y_layer, st = pu.run_layer(SMALL, layer, x, wfmt)
    assert st == 0
    assert np.array_equal(idx_l, idx_h)
    assert torch.equal(y, y_layer)


# ------------------------------------------------------------------ extreme e8m0 scales

NOSHARED = synth.LayerShape(hidden=512, n_experts=16, top_k=2, inter=128, shared_inter=0)


def _extreme_layer(big_in: bool):
    """MXFP4 layer whose expert block scales sit at the ends of the e8m0
    range. big_in: gate/up blocks at 2^126 / 2^127 (codes limited to
    magnitudes <= 1.5, so every weight is a finite fp32) and down blocks at
    2^-127, 2^-126, 2^-125 (scales 0, 1, 2; 2^-127 is an fp32 subnormal);
    otherwise the other way round. The tokens are scaled by 2^-100 or 2^100
    so that every intermediate value of the true result is a normal fp32."""
    layer = synth.device_layer(NOSHARED, 6, wfmt=1)
    lim = torch.tensor(0xBB, dtype=torch.uint8, device="cuda")  # keep sign and the two low bits per nibble

    def pattern(s, values):
        nb = s.shape[-1]
        v = torch.tensor(values, dtype=torch.uint8, device="cuda")
        return v[torch.arange(nb, device="cuda") % len(values)].expand_as(s).contiguous()

    big, small = [253, 254], [0, 1, 2]
    for n in ("1", "3"):
        layer["s" + n] = pattern(layer["s" + n], big if big_in else small)
        if big_in:
            layer["w" + n] = layer["w" + n] & lim
    layer["s2"] = pattern(layer["s2"], small if big_in else big)
    if not big_in:
        layer["w2"] = layer["w2"] & lim
    return layer


@pytest.mark.parametrize("big_in", [True, False])
@pytest.mark.parametrize("M", [1, 4])
def test_mxfp4_extreme_block_scales_in_the_fused_layer(api, big_in, M):
    layer = _extreme_layer(big_in)
    x = synth.x_independent(NOSHARED, 280 + M, M, device="cuda")
    e = -100 if big_in else 100
    xs = (x.float() * 2.0 ** e).to(torch.bfloat16)
    assert torch.equal(xs.float() * 2.0 ** -e, x.float())  # the scaling is exact
    err, _, _ = pu.compare_layer(NOSHARED, layer, xs, 1)
    # the expected output is finite and far from zero in both cases
    _, _, _, y_o = pu.oracle_layer(NOSHARED, layer, synth.to_u16(xs), 1)
    assert np.all(np.isfinite(y_o)) and np.linalg.norm(y_o.astype(np.float64)) > 0
