"""Helpers shared by the GPU parity tests: run the CUDA path through the
C ABI, run the oracle on the same seeded inputs, compare under the stated
tolerances.

Tolerances. Expert indices must match exactly, except for a token whose
oracle k-th and (k+1)-th logits differ by less than 1e-3 (then the GPU's
selection is checked for validity and its y is compared with the oracle run
on the GPU's own routing). Outputs: relative L2 error 1e-2 for bf16 and FP8 weights, 3e-2 for MXFP4
(each against the oracle on the same, dequantised, weights), over the whole
[M, H] block and for every token on its own.
Routing weights: 1e-4 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_decode_gb300 import synth

TIE_GAP = 1e-3
TOL_Y = {0: 1e-2, 1: 3e-2, 2: 1e-2}
TOL_W = 1e-4


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def bf16_bits_to_f32(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_to_f32(synth.to_u16(t))


def near_tie(logits_row: np.ndarray, k: int) -> bool:
    s = np.sort(logits_row.astype(np.float64))[::-1]
    return k < s.size and (s[k - 1] - s[k]) < TIE_GAP


def ranking_keys(logits: np.ndarray, router) -> np.ndarray:
    """What the router ranks: the logits (plain softmax router), else the
    scores (softmax or sigmoid) plus the selection bias."""
    if router is None or (router.get("scoring", 0) == 0 and router.get("bias") is None):
        return logits
    l = logits.astype(np.float64)
    if router.get("scoring", 0) == 1:
        s = 1.0 / (1.0 + np.exp(-l))
    else:
        e = np.exp(l - l.max(axis=1, keepdims=True))
        s = e / e.sum(axis=1, keepdims=True)
    b = router.get("bias")
    return s + (0.0 if b is None else b.cpu().numpy().astype(np.float64))


def check_routing(idx_gpu, w_gpu, idx_o, w_o, logits_o, k):
    """Returns the list of exempt (near-tie) tokens; asserts the rest."""
    exempt = []
    for t in range(idx_o.shape[0]):
        if near_tie(logits_o[t], k):
            exempt.append(t)
            assert len(set(idx_gpu[t])) == k and all(0 <= e < logits_o.shape[1] for e in idx_gpu[t])
            continue
        assert set(idx_gpu[t]) == set(idx_o[t]), (t, idx_gpu[t], idx_o[t])
        # order: only where adjacent selected logits are separated
        for j in range(k - 1):
            if logits_o[t, idx_o[t, j]] - logits_o[t, idx_o[t, j + 1]] >= TIE_GAP:
                assert idx_gpu[t, j] == idx_o[t, j], (t, j)
        wg = dict(zip(idx_gpu[t].tolist(), w_gpu[t].tolist()))
        for e, wv in zip(idx_o[t].tolist(), w_o[t].tolist()):
            assert abs(wg[e] - wv) <= TOL_W, (t, e, wg[e], wv)
    return exempt


def oracle_layer(shape, layer: dict, x_u16: np.ndarray, wfmt: int, idx_override=None, w_override=None,
                 router=None):
    """Oracle routing + FFN on host copies of the touched experts of a device
    layer. router: None (plain softmax) or a dict with scoring, bias (device
    fp32 [E] or None) and scale. Returns (idx, w, keys, y), keys being what
    the router ranks."""
    Wg = synth.to_u16(layer["Wg"])
    if router is None:
        idx, w, logits = oracle.route(x_u16, Wg, shape.top_k)
    else:
        b = router.get("bias")
        idx, w, logits = oracle.route_ex(x_u16, Wg, shape.top_k, scoring=router.get("scoring", 0),
                                         bias=None if b is None else b.cpu().numpy(),
                                         routed_scale=router.get("scale", 0.0))
    logits = ranking_keys(logits, router)
    ri = idx if idx_override is None else idx_override
    rw = w if w_override is None else w_override
    experts = {int(e): synth.host_expert(shape, layer, int(e), wfmt) for e in np.unique(ri)}
    shared = tuple(synth.to_u16(layer[n]) for n in ("ws1", "ws3", "ws2")) if shape.shared_inter else None
    y = oracle.ffn(x_u16, ri, rw, experts, shape.n_experts, shape.inter, shared, wfmt=wfmt)
    return idx, w, logits, y


def expert_weights_of(layer: dict, wfmt: int):
    """The layer's weights for the C ABI; a layer dict holding w2t (and ws2t)
    passes the transposed down projections too (split-K one-token layer)."""
    from moe_decode_gb300 import api
    return api.ExpertWeights(w1=layer["w1"], w3=layer["w3"], w2=layer["w2"], ws1=layer["ws1"],
                             ws3=layer["ws3"], ws2=layer["ws2"], s1=layer.get("s1"), s3=layer.get("s3"),
                             s2=layer.get("s2"), w2t=layer.get("w2t"), ws2t=layer.get("ws2t"))


def with_down_t(layer: dict) -> dict:
    """A copy of a bf16 layer dict with the transposed down projections
    (made by the library's moe_transpose_down)."""
    from moe_decode_gb300 import api
    d = dict(layer)
    d["w2t"] = api.transpose_down(layer["w2"])
    d["ws2t"] = api.transpose_down(layer["ws2"]) if layer["ws2"].numel() else None
    return d


def api_shape(shape, wfmt: int, router=None, io=None):
    from moe_decode_gb300 import api
    r = router or {}
    o = io or {}
    return api.make_shape(shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter, wfmt,
                          scoring=r.get("scoring", 0), routed_scale=r.get("scale", 0.0), router_bias=r.get("bias"),
                          norm_weight=o.get("gamma"), norm_eps=o.get("eps", 0.0), residual=o.get("residual", False))


def run_layer(shape, layer: dict, x: torch.Tensor, wfmt: int, flags: int = 0, router=None, io=None):
    """The fused layer through the C ABI. Returns (idx, w, y) on the host and
    the device status word."""
    from moe_decode_gb300 import api
    M = x.shape[0]
    s = api_shape(shape, wfmt, router, io)
    ws = api.workspace(s, M)
    idx = torch.full((M, shape.top_k), -1, dtype=torch.int32, device=x.device)
    w = torch.zeros((M, shape.top_k), dtype=torch.float32, device=x.device)
    y = torch.zeros((M, shape.hidden), dtype=torch.bfloat16, device=x.device)
    api.decode_layer(x, layer["Wg"], expert_weights_of(layer, wfmt), s, y, ws, idx, w, flags=flags)
    st = api.read_status(ws)
    return idx.cpu().numpy(), w.cpu().numpy(), y, st


def compare_layer(shape, layer, x: torch.Tensor, wfmt: int, router=None, io=None):
    """Full parity check of moe_decode_layer against the oracle. io: None or
    a dict with gamma (device bf16 [H]), eps and residual: the input x is
    then the residual stream, normalised by the oracle's RMSNorm, and the
    expected output includes the residual."""
    idx_g, w_g, y_g, st = run_layer(shape, layer, x, wfmt, router=router, io=io)
    assert st == 0, st
    return check_layer_output(shape, layer, x, idx_g, w_g, y_g, wfmt, router=router, io=io)


def check_layer_output(shape, layer, x: torch.Tensor, idx_g, w_g, y_g, wfmt: int, router=None, io=None):
    """Checks one call's routing (idx_g, w_g on the host) and output y_g (bf16
    tensor) against the oracle run on the call's own input x. Returns
    (rel L2 error, idx_g, exempt tokens)."""
    h_u16 = synth.to_u16(x)
    x_u16 = h_u16
    if io and io.get("gamma") is not None:
        eps = io.get("eps", 0.0)
        x_u16 = oracle.rmsnorm(h_u16, synth.to_u16(io["gamma"]), eps if eps > 0 else 1e-6)
    idx_o, w_o, logits_o, y_o = oracle_layer(shape, layer, x_u16, wfmt, router=router)
    exempt = check_routing(idx_g, w_g, idx_o, w_o, logits_o, shape.top_k)
    y_ref = y_o.copy()
    if exempt:
        _, _, _, y_alt = oracle_layer(shape, layer, x_u16, wfmt, idx_override=idx_g, w_override=w_g, router=router)
        y_ref[exempt] = y_alt[exempt]
    if io and io.get("residual"):
        y_ref = y_ref + oracle.bf16_to_f32(h_u16)
    y_gf = bf16_bits_to_f32(y_g)
    err = rel_l2(y_gf, y_ref)
    assert err <= TOL_Y[wfmt], err
    check_per_token(y_gf, y_ref, TOL_Y[wfmt])
    return err, idx_g, exempt


def check_per_token(y_gpu: np.ndarray, y_ref: np.ndarray, tol: float):
    """The tolerance holds for every token on its own, not only over the
    whole [M, H] block (one bad token cannot hide among good ones)."""
    for t in range(y_ref.shape[0]):
        e = rel_l2(y_gpu[t], y_ref[t])
        assert e <= tol, (t, e)
