"""Output layer (lm_head) and FP8 e4m3 helpers on the GPU against the
oracle: the e4m3 decode and the block quantiser bit for bit; logits within
a relative L2 error of 1e-5 (fp32 accumulation on both sides, in different
orders) on small ragged shapes and, for the 157,184 x 2,560 vocabulary, on
sampled rows whose weights the oracle quantises itself."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def api():
    from moe_decode_gb300 import build
    build.build()
    from moe_decode_gb300 import api as a
    oracle.build()
    a.set_option(a.OPT_GRID_CTAS, 0)
    a.set_option(a.OPT_WAIT_TIMEOUT_NS, 1_000_000_000)
    return a


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def lm_ws(api):
    ws = torch.empty(api.LM_HEAD_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    api.workspace_init(ws)
    return ws


def test_fp8_dequant_bit_exact(api):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(4, 1).cuda()   # [4, 256]
    scales = torch.tensor([[1.0, 0.5], [3.0, 2.0 ** -20], [0.013, 7.25], [1.0, 1.0]], dtype=torch.float32).cuda()
    out = torch.empty((4, 256), dtype=torch.float32, device="cuda")
    api.fp8_dequant(codes, scales, 128, out)
    got = out.cpu().numpy()
    sc = scales.cpu().numpy()
    for r in range(4):
        for c in range(256):
            want = np.float32(oracle.fp8_e4m3_value(c)) * sc[r, c // 128]
            g = got[r, c]
            assert (np.isnan(want) and np.isnan(g)) or g == want, (r, hex(c), g, want)


def test_fp8_quantize_bit_exact(api):
    R, K = 24, 512
    w = synth.normal_bf16(21, 1, 0, R * K, 0.02, "cuda").view(R, K).clone()
    w[3] = 0                                   # an all-zero row
    w[5, :7] = torch.tensor([-0.0, 1e-30, -1e-30, 3.0e38, -3.0e38, 1.0, -1.0], dtype=torch.bfloat16)
    w[7] *= 1e4
    for block in (32, 128, 512):
        codes = torch.empty((R, K), dtype=torch.uint8, device="cuda")
        scales = torch.empty((R, K // block), dtype=torch.float32, device="cuda")
        api.fp8_quantize(w, block, codes, scales)
        c_o, s_o = oracle.fp8_quantize(synth.to_u16(w), block)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), s_o.view(np.uint32)), block
        assert np.array_equal(codes.cpu().numpy(), c_o), block


def _run_lm(api, x, W, V, H, wfmt, scale=None):
    M = x.shape[0]
    logits = torch.full((M, V), float("nan"), dtype=torch.float32, device="cuda")
    ws = lm_ws(api)
    api.lm_head(x, W, V, H, logits, ws, wfmt=wfmt, w_scale=scale)
    assert api.read_status(ws) == 0
    return logits.cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 6, 9, 16])
@pytest.mark.parametrize("wfmt", [0, 2])
def test_lm_head_small_ragged(api, M, wfmt):
    """bf16 rows against three or more tokens run on the tensor cores."""
    V, H = 1000, 256                           # 1000 rows over 152 CTAs: uneven
    Wb = synth.normal_bf16(31, 1, 0, V * H, 0.02, "cuda").view(V, H)
    x = synth.normal_bf16(32 + M, 2, 0, M * H, 1.0, "cuda").view(M, H)
    if wfmt == 0:
        got = _run_lm(api, x, Wb, V, H, 0)
        want = oracle.lm_head(synth.to_u16(x), synth.to_u16(Wb), V)
    else:
        codes = torch.empty((V, H), dtype=torch.uint8, device="cuda")
        scales = torch.empty((V, 1), dtype=torch.float32, device="cuda")
        api.fp8_quantize(Wb, H, codes, scales)
        got = _run_lm(api, x, codes, V, H, 2, scales.view(V))
        c_o, s_o = oracle.fp8_quantize(synth.to_u16(Wb), H)
        want = oracle.lm_head(synth.to_u16(x), c_o, V, wfmt=2, scale=s_o[:, 0])
    assert np.isfinite(got).all()
    assert rel_l2(got, want) <= TOL


@pytest.mark.parametrize("wfmt", [0, 2])
def test_lm_head_token_scales(api, wfmt):
    """Tokens of very different magnitudes (and an all-zero one) in one call:
    FP8 launches hold each token in f16 times its own power of two, which must
    come back out of that token's logits, also within a token pair."""
    V, H, M = 700, 512, 5
    Wb = synth.normal_bf16(61, 1, 0, V * H, 0.02, "cuda").view(V, H)
    x = synth.normal_bf16(62, 2, 0, M * H, 1.0, "cuda").view(M, H).float()
    x[0] *= 1e-3
    x[1] *= 1e3
    x[2] = 0.0
    x[4] *= 37.0
    x = x.to(torch.bfloat16)
    if wfmt == 0:
        got = _run_lm(api, x, Wb, V, H, 0)
        want = oracle.lm_head(synth.to_u16(x), synth.to_u16(Wb), V)
    else:
        codes = torch.empty((V, H), dtype=torch.uint8, device="cuda")
        scales = torch.empty((V, 1), dtype=torch.float32, device="cuda")
        api.fp8_quantize(Wb, H, codes, scales)
        got = _run_lm(api, x, codes, V, H, 2, scales.view(V))
        c_o, s_o = oracle.fp8_quantize(synth.to_u16(Wb), H)
        want = oracle.lm_head(synth.to_u16(x), c_o, V, wfmt=2, scale=s_o[:, 0])
    assert np.all(got[2] == 0.0)
    for t in (0, 1, 3, 4):  # each token against its own reference
        assert rel_l2(got[t], want[t]) <= TOL, t


@pytest.mark.parametrize("M", [2, 5])
def test_lm_head_h_not_a_multiple_of_16(api, M):
    """H = 264 (a multiple of 8, not of 16): the CUDA-core path at any M."""
    V, H = 333, 264
    Wb = synth.normal_bf16(71, 1, 0, V * H, 0.02, "cuda").view(V, H)
    x = synth.normal_bf16(72 + M, 2, 0, M * H, 1.0, "cuda").view(M, H)
    got = _run_lm(api, x, Wb, V, H, 0)
    assert rel_l2(got, oracle.lm_head(synth.to_u16(x), synth.to_u16(Wb), V)) <= TOL


def test_lm_head_fewer_rows_than_ctas(api):
    V, H, M = 7, 512, 5
    Wb = synth.normal_bf16(41, 1, 0, V * H, 0.02, "cuda").view(V, H)
    x = synth.normal_bf16(42, 2, 0, M * H, 1.0, "cuda").view(M, H)
    got = _run_lm(api, x, Wb, V, H, 0)
    assert rel_l2(got, oracle.lm_head(synth.to_u16(x), synth.to_u16(Wb), V)) <= TOL


@pytest.mark.parametrize("wfmt,M", [(0, 2), (2, 2), (0, 6)])
def test_lm_head_full_vocabulary_sampled_rows(api, wfmt, M):
    V, H = 157184, 2560
    Wb = synth.normal_bf16(51, 1, 0, V * H, 0.02, "cuda").view(V, H)
    x = synth.normal_bf16(52, 2, 0, M * H, 1.0, "cuda").view(M, H)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(V - 8, V),
                                     np.random.default_rng(0).integers(0, V, 240)]))
    Ws = synth.to_u16(Wb[torch.from_numpy(rows).cuda()])
    if wfmt == 0:
        got = _run_lm(api, x, Wb, V, H, 0)
        want = oracle.lm_head(synth.to_u16(x), Ws, len(rows))
    else:
        codes = torch.empty((V, H), dtype=torch.uint8, device="cuda")
        scales = torch.empty((V, 1), dtype=torch.float32, device="cuda")
        api.fp8_quantize(Wb, H, codes, scales)
        del Wb
        got = _run_lm(api, x, codes, V, H, 2, scales.view(V))
        c_o, s_o = oracle.fp8_quantize(Ws, H)
        want = oracle.lm_head(synth.to_u16(x), c_o, len(rows), wfmt=2, scale=s_o[:, 0])
    assert np.isfinite(got).all()
    assert rel_l2(got[:, rows], want) <= TOL
    torch.cuda.empty_cache()
