"""moe_decode_layer_static_scratch: the layer without a caller workspace.

Its scratch is a fixed device array of the library, so it is checked here,
in the file pytest collects last, after every other test has run with its
own workspaces. The GPU tests compare it bit for bit with moe_decode_layer
(same kernel and launch configuration, fixed-order accumulation) on two
calls in a row, and check that repeated calls leave the device's free
memory unchanged. The host-side size check needs no GPU.
"""
import ctypes

import pytest
import torch

from moe_decode_gb300 import synth


@pytest.fixture(scope="module")
def api():
    from moe_decode_gb300 import build
    build.build()
    from moe_decode_gb300 import api as a
    return a


def test_rejects_shapes_beyond_the_static_scratch(api):
    big = api.make_shape(8192, 1024, 16, 4096, 4096, 0)
    assert api.workspace_bytes(big, 16) > api.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(4096)
    w = api._Weights(4096, 4096, 4096, None, None, None, 4096, 4096, 4096)
    rc = api.lib.moe_decode_layer_static_scratch(fake, 16, fake, ctypes.byref(w), ctypes.byref(big), None, None,
                                                 fake, 0, None)
    assert rc == api.ESCRATCH
    assert "static scratch" in api.status_str(rc)
    assert api.last_launch_count() == 0
    ling = api.make_shape(2560, 512, 8, 768, 768, 0)
    assert api.workspace_bytes(ling, 16) <= api.STATIC_SCRATCH_BYTES
    assert api.lib.moe_decode_layer_static_scratch(fake, 1, fake, ctypes.byref(w), ctypes.byref(ling), None, None,
                                                   fake, 1 << 4, None) == api.EINVAL   # unknown flag


def _run_pair(api, layer, shape, wfmt, x, flags=0):
    """Both entry points on the same inputs; returns their (idx, w, y)."""
    from parity_util import expert_weights_of
    M = x.shape[0]
    s = api.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter, wfmt)
    ew = expert_weights_of(layer, wfmt)
    outs = []
    for static in (False, True):
        idx = torch.full((M, shape.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((M, shape.top_k), dtype=torch.float32, device="cuda")
        y = torch.zeros((M, shape.hidden), dtype=torch.bfloat16, device="cuda")
        if static:
            api.decode_layer_static_scratch(x, layer["Wg"], ew, s, y, idx, w, flags=flags)
        else:
            ws = api.workspace(s, M)
            api.decode_layer(x, layer["Wg"], ew, s, y, ws, idx, w)
            assert api.read_status(ws) == 0
        torch.cuda.synchronize()
        outs.append((idx, w, y))
    return outs


@pytest.mark.gpu
@pytest.mark.parametrize("wfmt", [0, 1, 2])
def test_matches_decode_layer_on_two_calls_in_a_row(api, wfmt):
    api.set_option(api.OPT_GRID_CTAS, 0)
    api.set_option(api.OPT_WAIT_TIMEOUT_NS, 1_000_000_000)
    layer = synth.device_layer(synth.LING, 0, wfmt=wfmt)
    for call, M in enumerate((6, 6)):
        x = synth.x_independent(synth.LING, 40 + call, M, device="cuda")
        (i0, w0, y0), (i1, w1, y1) = _run_pair(api, layer, synth.LING, wfmt, x)
        assert api.last_launch_count() == 1
        assert torch.equal(i0, i1), call
        assert torch.equal(w0, w1), call
        assert torch.equal(y0, y1), call
    del layer
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_allocates_nothing_and_resets(api):
    api.set_option(api.OPT_GRID_CTAS, 0)
    layer = synth.device_layer(synth.TINY, 0)
    from parity_util import expert_weights_of
    sh = synth.TINY
    s = api.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.inter, sh.shared_inter, 0)
    ew = expert_weights_of(layer, 0)
    xs = [synth.x_independent(sh, 60 + i, 16, device="cuda") for i in range(4)]
    ys = [torch.zeros((16, sh.hidden), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    api.decode_layer_static_scratch(xs[0], layer["Wg"], ew, s, ys[0])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for i in (1, 2, 3):
        api.decode_layer_static_scratch(xs[i], layer["Wg"], ew, s, ys[i],
                                        flags=api.F_RESET_SCRATCH if i == 2 else 0)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    (_, _, y_ref), (_, _, y_static) = _run_pair(api, layer, sh, 0, xs[3])
    assert torch.equal(ys[3], y_ref)
    assert torch.equal(y_static, y_ref)
    (_, _, y_ref2), _ = _run_pair(api, layer, sh, 0, xs[2])
    assert torch.equal(ys[2], y_ref2)


@pytest.mark.gpu
def test_timeout_is_reported_sticky_and_cleared_by_reset(api):
    """A bounded device wait forced to run out (a 2 ms budget) is reported
    through moe_static_scratch_status; the next plain call refuses to run
    (its output stays untouched and the status stays MOE_ETIMEOUT) instead of
    computing on stale control words; a call with MOE_F_RESET_SCRATCH then
    matches moe_decode_layer bit for bit."""
    from parity_util import expert_weights_of
    api.set_option(api.OPT_GRID_CTAS, 0)
    sh = synth.TINY
    layer = synth.device_layer(sh, 0)
    ew = expert_weights_of(layer, 0)
    s = api.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.inter, sh.shared_inter, 0)
    x = synth.x_independent(sh, 70, 3, device="cuda")
    y = torch.zeros((3, sh.hidden), dtype=torch.bfloat16, device="cuda")
    api.set_option(api.OPT_WAIT_TIMEOUT_NS, 2_000_000)
    try:
        api.decode_layer_static_scratch(x, layer["Wg"], ew, s, y, flags=api.F_DEBUG_FORCE_TIMEOUT)
        assert api.static_scratch_status() == api.ETIMEOUT
    finally:
        api.set_option(api.OPT_WAIT_TIMEOUT_NS, 1_000_000_000)
    y_stale = torch.full_like(y, 7.0)
    api.decode_layer_static_scratch(x, layer["Wg"], ew, s, y_stale)
    assert api.static_scratch_status() == api.ETIMEOUT
    assert torch.equal(y_stale, torch.full_like(y, 7.0))
    api.decode_layer_static_scratch(x, layer["Wg"], ew, s, y, flags=api.F_RESET_SCRATCH)
    assert api.static_scratch_status() == 0
    (_, _, y_ref), _ = _run_pair(api, layer, sh, 0, x)
    assert torch.equal(y, y_ref)
