"""Seeded synthetic inputs for the MoE decode layer.

This module generates weights and activations only. It holds none of the
layer's arithmetic: no routing, activation, projection or combine step.
Both the CUDA path (benchmark, tests) and the CPU oracle (tests) take
their inputs from here.

Generator. Every element is a pure function of (seed, tensor id, flat element
index): two 32-bit integer hashes of the counter give four 16-bit uniforms, whose
sum (Irwin-Hall, n = 4) is centred and scaled to mean 0 and standard deviation
sigma. All steps are integer operations, one exact int -> fp32 conversion, one
fp32 multiply and one round-to-nearest-even cast to bf16, so the same element
has the same bits on the CPU and on the GPU, on any torch version. Any slice of
a tensor (one expert's matrix, say) can be generated on its own.

The tails stop at +-2*sqrt(3)*sigma; the mean, the variance and the
near-Gaussian shape match the N(0, 0.02) weights and N(0, 1) activations of
the workloads this layer is measured on.

MXFP4 weights are the bf16 draws quantised block by block (32 elements along
the reduction dimension): e8m0 scale E = clamp(floor(log2 amax) - 2 + 127,
0, 254) (0 for an all-zero block), e2m1 codes by round-to-nearest-even of
w / 2^(E-127), saturating at 6, element 2j in the low nibble of byte j.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

M32 = 0xFFFFFFFF
_MUL = 0x45D9F3B
CHUNK = 1 << 24

# tensor ids of the generator streams
T_WG, T_W1, T_W3, T_W2, T_WS1, T_WS3, T_WS2, T_X, T_XU = range(1, 10)

WEIGHT_SIGMA = 0.02
X_SIGMA = 1.0
LAYER_SEED0 = 1000  # layer copy c uses seed 1000 + c
X_SEED0 = 2000      # input of step s uses seed 2000 + s

# Shared-component weight for the ~50% consecutive-overlap input recipe of the
# M = 10 verify-block workload: x_t = sqrt(rho) u + sqrt(1 - rho) z_t. Derived
# by tests/golden/derive_overlap_rho.py (oracle router on layer copy 0) and
# recorded with its measured overlap in tests/golden/overlap_rho.json.
RHO_OVERLAP_M10 = 0.8759765625


def _mix_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * _MUL) & M32
    x ^= x >> 16
    x = (x * _MUL) & M32
    x ^= x >> 16
    return x


def _mix(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    return x


def _keys(seed: int, tid: int):
    base = _mix_int(_mix_int(seed) ^ _mix_int(tid * 0x9E3779B1))
    return _mix_int(base ^ 0x68E31DA4), _mix_int(base ^ 0xB5297A4D)


def normal_f32(seed: int, tid: int, start: int, count: int, sigma: float,
               device="cpu") -> torch.Tensor:
    """Elements [start, start+count) of stream (seed, tid) as fp32."""
    if start < 0 or start + count > (1 << 32):
        raise ValueError("a generator stream holds at most 2^32 elements")
    k1, k2 = _keys(seed, tid)
    scale = torch.tensor(np.float32(sigma * math.sqrt(3.0) / 65536.0), device=device)
    out = torch.empty(count, dtype=torch.float32, device=device)
    for c0 in range(0, count, CHUNK):
        n = min(CHUNK, count - c0)
        i = torch.arange(start + c0, start + c0 + n, dtype=torch.int64, device=device)
        a = _mix(i ^ k1)
        b = _mix(i ^ k2)
        s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)
        out[c0:c0 + n] = (s - 131070).to(torch.float32) * scale
    return out


def normal_bf16(seed: int, tid: int, start: int, count: int, sigma: float,
                device="cpu") -> torch.Tensor:
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    for c0 in range(0, count, CHUNK):
        n = min(CHUNK, count - c0)
        out[c0:c0 + n] = normal_f32(seed, tid, start + c0, n, sigma, device).to(torch.bfloat16)
    return out


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int

    @property
    def expert_bytes_bf16(self) -> int:
        return 3 * self.hidden * self.inter * 2

    @property
    def shared_bytes(self) -> int:
        return 3 * self.hidden * self.shared_inter * 2

    @property
    def router_bytes(self) -> int:
        return self.n_experts * self.hidden * 2


TINY = LayerShape(hidden=256, n_experts=16, top_k=2, inter=64, shared_inter=64)
LING = LayerShape(hidden=2560, n_experts=512, top_k=8, inter=768, shared_inter=768)


# ---------------------------------------------------------------------------
# weights

def router_weight(shape: LayerShape, copy: int, device="cpu") -> torch.Tensor:
    E, H = shape.n_experts, shape.hidden
    return normal_bf16(LAYER_SEED0 + copy, T_WG, 0, E * H, WEIGHT_SIGMA, device).view(E, H)


def expert_weights(shape: LayerShape, copy: int, e: int, device="cpu"):
    """(W1 [I,H], W3 [I,H], W2 [H,I]) bf16 of routed expert e, as a slice of
    the full [E, ...] streams (identical to the same slice of the full tensor)."""
    H, I = shape.hidden, shape.inter
    n = I * H
    seed = LAYER_SEED0 + copy
    w1 = normal_bf16(seed, T_W1, e * n, n, WEIGHT_SIGMA, device).view(I, H)
    w3 = normal_bf16(seed, T_W3, e * n, n, WEIGHT_SIGMA, device).view(I, H)
    w2 = normal_bf16(seed, T_W2, e * n, n, WEIGHT_SIGMA, device).view(H, I)
    return w1, w3, w2


def shared_weights(shape: LayerShape, copy: int, device="cpu"):
    H, Is = shape.hidden, shape.shared_inter
    n = Is * H
    seed = LAYER_SEED0 + copy
    ws1 = normal_bf16(seed, T_WS1, 0, n, WEIGHT_SIGMA, device).view(Is, H)
    ws3 = normal_bf16(seed, T_WS3, 0, n, WEIGHT_SIGMA, device).view(Is, H)
    ws2 = normal_bf16(seed, T_WS2, 0, n, WEIGHT_SIGMA, device).view(H, Is)
    return ws1, ws3, ws2


def all_expert_weights(shape: LayerShape, copy: int, device="cpu"):
    """Full routed tensors (W1 [E,I,H], W3 [E,I,H], W2 [E,H,I]) bf16."""
    E, H, I = shape.n_experts, shape.hidden, shape.inter
    seed = LAYER_SEED0 + copy
    n = E * I * H
    w1 = normal_bf16(seed, T_W1, 0, n, WEIGHT_SIGMA, device).view(E, I, H)
    w3 = normal_bf16(seed, T_W3, 0, n, WEIGHT_SIGMA, device).view(E, I, H)
    w2 = normal_bf16(seed, T_W2, 0, n, WEIGHT_SIGMA, device).view(E, H, I)
    return w1, w3, w2


# ---------------------------------------------------------------------------
# MXFP4 encoding of synthetic weights

def mxfp4_quantize(w: torch.Tensor):
    """bf16/fp32 [..., K] -> (codes uint8 [..., K/2], scales uint8 [..., K/32])."""
    K = w.shape[-1]
    assert K % 32 == 0
    lead = w.shape[:-1]
    v = w.to(torch.float32).reshape(-1, K // 32, 32)
    amax = v.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)                  # amax = m * 2^ex, m in [0.5, 1)
    E = (ex.to(torch.int32) - 1) - 2 + 127     # floor(log2 amax) - emax(e2m1) + bias
    E = torch.clamp(E, 0, 254)
    E = torch.where(amax == 0, torch.zeros_like(E), E)
    # 2^(127 - E) built from its bit pattern (exact; E = 254 gives the
    # subnormal 2^-127)
    bits = torch.where(E < 254, (254 - E) << 23, torch.full_like(E, 1 << 22))
    a = v * bits.view(torch.float32).unsqueeze(-1)
    mag = a.abs()
    # round to nearest, ties to the even code, on {0,.5,1,1.5,2,3,4,6}
    code = ((mag > 0.25).to(torch.int32) + (mag >= 0.75).to(torch.int32)
            + (mag > 1.25).to(torch.int32) + (mag >= 1.75).to(torch.int32)
            + (mag > 2.5).to(torch.int32) + (mag >= 3.5).to(torch.int32)
            + (mag > 5.0).to(torch.int32))
    code = code + torch.where((a < 0) & (code > 0), 8, 0).to(torch.int32)
    code = code.reshape(-1, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).to(torch.uint8)
    return packed.reshape(*lead, K // 2), E.to(torch.uint8).reshape(*lead, K // 32)


# ---------------------------------------------------------------------------
# FP8 e4m3 encoding of synthetic weights

FP8_BLOCK = 128


def fp8_quantize(w: torch.Tensor, block: int = FP8_BLOCK):
    """bf16/fp32 [..., K] -> (e4m3 codes uint8 [..., K], fp32 scales
    [..., K / block]): scale = amax(block) / 448 in fp32 (1 for an all-zero
    block), code = the e4m3 value nearest to w / scale (torch's float8
    conversion: round to nearest even; the quotient never exceeds 448 by
    more than a rounding error, and is clamped to +-448 first)."""
    K = w.shape[-1]
    assert K % block == 0
    lead = w.shape[:-1]
    v = w.to(torch.float32).reshape(-1, K // block, block)
    amax = v.abs().amax(dim=-1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = torch.clamp(v / sc.unsqueeze(-1), -448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.reshape(*lead, K), sc.reshape(*lead, K // block)


# ---------------------------------------------------------------------------
# activations

def x_independent(shape: LayerShape, step: int, M: int, device="cpu") -> torch.Tensor:
    """M tokens drawn independently: x [M, H] bf16 ~ N(0, 1)."""
    H = shape.hidden
    return normal_bf16(X_SEED0 + step, T_X, 0, M * H, X_SIGMA, device).view(M, H)


def x_overlap(shape: LayerShape, step: int, M: int, rho: float = RHO_OVERLAP_M10,
              device="cpu") -> torch.Tensor:
    """x_t = sqrt(rho) u + sqrt(1 - rho) z_t with u shared by the step's tokens
    and z_t per token, all ~N(0, 1), rounded once to bf16. The router is linear
    in x, so this gives each token's logits a shared per-step component plus
    per-token noise."""
    H = shape.hidden
    u = normal_f32(X_SEED0 + step, T_XU, 0, H, X_SIGMA, device).view(1, H)
    z = normal_f32(X_SEED0 + step, T_X, 0, M * H, X_SIGMA, device).view(M, H)
    c1 = torch.tensor(np.float32(math.sqrt(rho)), device=device)
    c2 = torch.tensor(np.float32(math.sqrt(1.0 - rho)), device=device)
    a = u * c1
    b = z * c2
    return (a + b).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# whole layers on the device

def device_layer(shape: LayerShape, copy: int, wfmt: int = 0, device="cuda") -> dict:
    """All weights of layer copy `copy`, generated on `device`.

    Keys: Wg, ws1, ws3, ws2 (bf16) and, for wfmt 0, w1, w3, w2 (bf16
    [E,I,H], [E,I,H], [E,H,I]); for wfmt 1, w1, w3, w2 as MXFP4 codes with
    s1, s3, s2 scales; for wfmt 2, as FP8 e4m3 codes with fp32 scales per 128
    elements (the bf16 draws quantised, expert block by block)."""
    d = {"Wg": router_weight(shape, copy, device)}
    d["ws1"], d["ws3"], d["ws2"] = shared_weights(shape, copy, device)
    E, H, I = shape.n_experts, shape.hidden, shape.inter
    seed = LAYER_SEED0 + copy
    n = I * H
    if wfmt == 0:
        d["w1"], d["w3"], d["w2"] = all_expert_weights(shape, copy, device)
        return d
    blk = max(1, (1 << 24) // n)
    for name, tid, rows, K in (("w1", T_W1, I, H), ("w3", T_W3, I, H), ("w2", T_W2, H, I)):
        if wfmt == 1:
            codes = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=device)
            scales = torch.empty((E, rows, K // 32), dtype=torch.uint8, device=device)
        else:
            codes = torch.empty((E, rows, K), dtype=torch.uint8, device=device)
            scales = torch.empty((E, rows, K // FP8_BLOCK), dtype=torch.float32, device=device)
        for e0 in range(0, E, blk):
            e1 = min(E, e0 + blk)
            w = normal_bf16(seed, tid, e0 * n, (e1 - e0) * n, WEIGHT_SIGMA, device).view(e1 - e0, rows, K)
            codes[e0:e1], scales[e0:e1] = mxfp4_quantize(w) if wfmt == 1 else fp8_quantize(w)
        d[name] = codes
        d["s" + name[1]] = scales
    return d


def host_expert(shape: LayerShape, layer: dict, e: int, wfmt: int = 0):
    """Host (numpy) copies of expert e's weights from a device layer, in the
    tuple order the CPU oracle takes."""
    if wfmt == 0:
        return tuple(to_u16(layer[n][e]) for n in ("w1", "w3", "w2"))
    return tuple(layer[n][e].cpu().numpy() for n in ("w1", "s1", "w3", "s3", "w2", "s2"))
