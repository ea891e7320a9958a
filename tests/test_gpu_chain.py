"""Consecutive layers chained with programmatic dependent launch: L calls of
moe_decode_layer issued back to back on one stream, on one workspace, the
output of call n being the input of call n + 1, with no synchronisation in
between. Each launch starts its prologue (weight tiles, and the router bias)
while the previous one still runs and must wait for it before reading its
output or rewriting the workspace ("Chasing the Batch-1 Floor", section
"PDL: stacking the latency floors of small kernels": the early trigger is
safe only if every consumer waits before each read of producer output).

Every layer's output is checked against the oracle run on that layer's own
input, and a ping-pong chain (call n + 1 writes the buffer call n reads) must
give the same bits as the chain with a buffer per layer."""
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


def _chain(api, shapes, layers, wfmt, x0, io, ws, pingpong: bool):
    """Issues the whole chain without synchronising; returns the input of
    every layer and the last output (device tensors), and the routing."""
    M, H = x0.shape
    k = shapes[0].top_k
    if pingpong:
        bufs = [x0.clone(), torch.zeros_like(x0)]
    else:
        bufs = [x0.clone()] + [torch.zeros_like(x0) for _ in shapes]
    idx = [torch.full((M, k), -1, dtype=torch.int32, device="cuda") for _ in shapes]
    w = [torch.zeros((M, k), dtype=torch.float32, device="cuda") for _ in shapes]
    ins = []
    for n, (sh, L) in enumerate(zip(shapes, layers)):
        src = bufs[n % 2] if pingpong else bufs[n]
        dst = bufs[(n + 1) % 2] if pingpong else bufs[n + 1]
        if not pingpong:
            ins.append(src)
        s = pu.api_shape(sh, wfmt, io=io[n] if io else None)
        api.decode_layer(src, L["Wg"], pu.expert_weights_of(L, wfmt), s, dst, ws, idx[n], w[n])
    out = bufs[len(shapes) % 2] if pingpong else bufs[-1]
    return ins, out, idx, w


def _run_and_check(api, shapes, layers, wfmt, x0, io=None):
    M = x0.shape[0]
    nbytes = max(api.workspace_bytes(pu.api_shape(sh, wfmt), M) for sh in shapes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    api.workspace_init(ws)
    ins, out, idx, w = _chain(api, shapes, layers, wfmt, x0, io, ws, pingpong=False)
    assert api.read_status(ws) == 0
    outs = ins[1:] + [out]
    for n, sh in enumerate(shapes):
        pu.check_layer_output(sh, layers[n], ins[n], idx[n].cpu().numpy(), w[n].cpu().numpy(), outs[n], wfmt,
                              io=io[n] if io else None)
    # the same chain on two buffers, reusing the same workspace
    _, out_pp, _, _ = _chain(api, shapes, layers, wfmt, x0, io, ws, pingpong=True)
    assert api.read_status(ws) == 0
    assert torch.equal(out_pp, out)


TINY_IS = [64, 128, 0, 192, 64, 128]


def _tiny_chain():
    shapes = [synth.LayerShape(256, 16, 2, 64, Is) for Is in TINY_IS]
    layers = [synth.device_layer(sh, 10 + n) for n, sh in enumerate(shapes)]
    return shapes, layers


@pytest.mark.parametrize("M", [1, 5, 16])
def test_tiny_chain_of_six_layers(api, M):
    shapes, layers = _tiny_chain()
    x0 = synth.x_independent(shapes[0], 300 + M, M, device="cuda")
    _run_and_check(api, shapes, layers, 0, x0)


@pytest.mark.parametrize("M", [1, 7])
def test_tiny_chain_with_norm_and_residual(api, M):
    """The chain as a model runs it: each layer reads the residual stream,
    normalises it with its own weight and adds its output to it."""
    shapes, layers = _tiny_chain()
    io = [dict(gamma=synth.normal_bf16(320 + n, 8, 0, 256, 1.0, "cuda"), eps=1e-6, residual=True)
          for n in range(len(shapes))]
    h0 = synth.normal_bf16(330 + M, 9, 0, M * 256, 3.0, "cuda").view(M, 256)
    _run_and_check(api, shapes, layers, 0, h0, io=io)


@pytest.mark.parametrize("wfmt", [0, 1])
def test_ling_chain_of_four_layers(api, wfmt):
    shapes = [synth.LING] * 4
    layers = [synth.device_layer(synth.LING, n, wfmt=wfmt) for n in range(2)]
    layers = layers + layers  # two copies, each used twice
    x0 = synth.x_independent(synth.LING, 340 + wfmt, 6, device="cuda")
    _run_and_check(api, shapes, layers, wfmt, x0)
    del layers
    torch.cuda.empty_cache()


def test_mixed_calls_on_one_workspace(api):
    """Routing-only, FFN-only, one-token (two-phase and split-K) and
    multi-token layer calls alternate on one workspace, issued back to back
    without synchronising. The calls share the workspace's control words: a
    call with an FFN uses the barrier and work counter of its epoch's parity
    and advances the epoch once its grid barrier has passed, a routing-only
    call advances it at exit. Every call is checked against the oracle."""
    sh = synth.TINY
    L = pu.with_down_t(synth.device_layer(sh, 21))
    s = pu.api_shape(sh, 0)
    k = sh.top_k
    nbytes = max(api.workspace_bytes(s, m) for m in (1, 6))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    api.workspace_init(ws)
    W = pu.expert_weights_of(L, 0)
    W2 = pu.expert_weights_of({n: v for n, v in L.items() if n not in ("w2t", "ws2t")}, 0)
    plan = ["route", "layer", "ffn", "splitk", "route", "layer", "layer", "route", "splitk", "layer", "ffn", "splitk"]
    Ms = [3, 1, 5, 1, 1, 6, 1, 2, 1, 2, 4, 1]
    ffn_idx = {}
    calls = []
    for n, (kind, M) in enumerate(zip(plan, Ms)):
        x = synth.x_independent(sh, 700 + n, M, device="cuda")
        idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((M, k), dtype=torch.float32, device="cuda")
        y = torch.zeros((M, sh.hidden), dtype=torch.bfloat16, device="cuda")
        if kind == "route":
            api.route(x, L["Wg"], s, idx, w, ws)
        elif kind == "ffn":
            rng = np.random.default_rng(800 + n)
            ih = np.stack([rng.choice(sh.n_experts, k, replace=False) for _ in range(M)]).astype(np.int32)
            wh = rng.uniform(0.1, 1.0, (M, k)).astype(np.float32)
            ffn_idx[n] = (ih, wh)
            idx.copy_(torch.from_numpy(ih))
            w.copy_(torch.from_numpy(wh))
            api.ffn(x, idx, w, W2, s, y, ws)
        else:
            api.decode_layer(x, L["Wg"], W if kind == "splitk" else W2, s, y, ws, idx, w)
        calls.append((kind, x, idx, w, y))
    torch.cuda.synchronize()
    assert api.read_status(ws) == 0
    for n, (kind, x, idx, w, y) in enumerate(calls):
        xu = synth.to_u16(x)
        if kind == "route":
            idx_o, w_o, logits_o = oracle.route(xu, synth.to_u16(L["Wg"]), k)
            pu.check_routing(idx.cpu().numpy(), w.cpu().numpy(), idx_o, w_o, logits_o, k)
        elif kind == "ffn":
            ih, wh = ffn_idx[n]
            _, _, _, y_o = pu.oracle_layer(sh, L, xu, 0, idx_override=ih, w_override=wh)
            yg = pu.bf16_bits_to_f32(y)
            assert pu.rel_l2(yg, y_o) <= pu.TOL_Y[0]
            pu.check_per_token(yg, y_o, pu.TOL_Y[0])
        else:
            pu.check_layer_output(sh, L, x, idx.cpu().numpy(), w.cpu().numpy(), y, 0)
