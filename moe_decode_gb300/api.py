"""Python binding of libmoe_decode.so (ctypes). Argument marshalling only:
every step of the layer runs in the library's CUDA kernels. Tensors are
torch CUDA tensors; their device pointers and the current stream are passed
through the C ABI declared in include/moe_decode.h.

There is no fallback: if the compiled library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_decode.so")

OK = 0
EINVAL, ESHAPE, EM, EWORKSPACE, EALIGN, ECUDA, ENODEVICE, ESCRATCH = -1, -2, -3, -4, -5, -6, -7, -8
EDEVICE_BAD_INDEX, ETIMEOUT = -100, -101
F_NO_PDL = 1
F_RESET_SCRATCH = 2
F_DEBUG_FORCE_TIMEOUT = 256
OPT_GRID_CTAS = 1
OPT_WAIT_TIMEOUT_NS = 2
OPT_TRACE_BUFFER = 3
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
LM_HEAD_WORKSPACE_BYTES = 1024
STATIC_SCRATCH_BYTES = 524288


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({status_str(code)})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("shared_inter", ctypes.c_int32), ("wfmt", ctypes.c_int32),
                ("scoring", ctypes.c_int32), ("routed_scale", ctypes.c_float), ("router_bias", ctypes.c_void_p),
                ("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float), ("residual", ctypes.c_int32)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1", "w3", "w2", "s1", "s3", "s2", "ws1", "ws3", "ws2", "w2t",
                                                 "ws2t")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m moe_decode_gb300.build` "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sp = ctypes.POINTER(Shape)
    wp = ctypes.POINTER(_Weights)
    lib.moe_workspace_bytes.argtypes = [sp, I32]
    lib.moe_workspace_bytes.restype = SZ
    lib.moe_workspace_init.argtypes = [P, SZ, P]
    lib.moe_route.argtypes = [P, I32, P, sp, P, P, P, SZ, P]
    lib.moe_ffn.argtypes = [P, I32, P, P, wp, sp, P, P, SZ, P]
    lib.moe_decode_layer.argtypes = [P, I32, P, wp, sp, P, P, P, P, SZ, ctypes.c_uint32, P]
    lib.moe_decode_layer_static_scratch.argtypes = [P, I32, P, wp, sp, P, P, P, ctypes.c_uint32, P]
    lib.moe_read_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_static_scratch_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_status_str.argtypes = [I32]
    lib.moe_status_str.restype = ctypes.c_char_p
    lib.moe_mxfp4_dequant.argtypes = [P, P, I64, I32, P, P]
    lib.moe_set_option.argtypes = [I32, I64]
    lib.moe_lm_head.argtypes = [P, I32, P, P, I32, I32, I32, P, P, SZ, ctypes.c_uint32, P]
    lib.moe_fp8_quantize.argtypes = [P, I64, I32, I32, P, P, P]
    lib.moe_fp8_dequant.argtypes = [P, P, I64, I32, I32, P, P]
    lib.moe_transpose_down.argtypes = [P, I64, I32, I32, P, P]
    lib.moe_last_launch_count.argtypes = []
    for f in ("moe_workspace_init", "moe_route", "moe_ffn", "moe_decode_layer", "moe_decode_layer_static_scratch",
              "moe_read_status", "moe_static_scratch_status", "moe_mxfp4_dequant", "moe_set_option", "moe_last_launch_count",
              "moe_lm_head", "moe_fp8_quantize", "moe_fp8_dequant", "moe_transpose_down"):
        getattr(lib, f).restype = I32
    return lib


lib = _load()


def status_str(code: int) -> str:
    return lib.moe_status_str(code).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise MoeError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(hidden, n_experts, top_k, inter, shared_inter, wfmt=0, scoring: int = 0, routed_scale: float = 0.0,
               router_bias: Optional[torch.Tensor] = None, norm_weight: Optional[torch.Tensor] = None,
               norm_eps: float = 0.0, residual: bool = False) -> Shape:
    """Layer shape, router configuration and input/output options;
    router_bias (fp32 [E]) and norm_weight (bf16 [H]) are device tensors that
    must stay alive while the shape is used."""
    return Shape(hidden, n_experts, top_k, inter, shared_inter, wfmt, scoring, routed_scale,
                 None if router_bias is None else router_bias.data_ptr(),
                 None if norm_weight is None else norm_weight.data_ptr(), norm_eps, int(residual))


@dataclass
class ExpertWeights:
    """Device tensors of one layer's experts (layouts in include/moe_decode.h).
    bf16: w1, w3 [E,I,H], w2 [E,H,I]; MXFP4: w1, w3 u8 [E,I,H/2], s1, s3 u8
    [E,I,H/32], w2 u8 [E,H,I/2], s2 u8 [E,H,I/32]; FP8: w1, w3 u8 [E,I,H],
    s1, s3 fp32 [E,I,H/128], w2 u8 [E,H,I], s2 fp32 [E,H,I/128]. Shared
    expert bf16."""
    w1: torch.Tensor
    w3: torch.Tensor
    w2: torch.Tensor
    ws1: Optional[torch.Tensor] = None
    ws3: Optional[torch.Tensor] = None
    ws2: Optional[torch.Tensor] = None
    s1: Optional[torch.Tensor] = None
    s3: Optional[torch.Tensor] = None
    s2: Optional[torch.Tensor] = None
    w2t: Optional[torch.Tensor] = None   # bf16 [E, I, H] (transpose_down(w2)); one-token split-K layer
    ws2t: Optional[torch.Tensor] = None  # bf16 [Is, H]

    def cstruct(self) -> _Weights:
        return _Weights(*(None if t is None else t.data_ptr() for t in
                          (self.w1, self.w3, self.w2, self.s1, self.s3, self.s2, self.ws1, self.ws3, self.ws2,
                           self.w2t, self.ws2t)))


def workspace_bytes(shape: Shape, M: int) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(shape), M))


def workspace_init(ws: torch.Tensor, stream=None):
    _check(lib.moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def workspace(shape: Shape, M: int, device="cuda", stream=None) -> torch.Tensor:
    n = workspace_bytes(shape, M)
    if n == 0:
        raise MoeError(ESHAPE, "moe_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def route(x, Wg, shape: Shape, idx, w, ws, stream=None):
    _check(lib.moe_route(_ptr(x), x.shape[0], _ptr(Wg), ctypes.byref(shape), _ptr(idx), _ptr(w), _ptr(ws),
                         ws.numel(), _stream(stream)), "moe_route")


def ffn(x, idx, w, weights: ExpertWeights, shape: Shape, y, ws, stream=None):
    cw = weights.cstruct()
    _check(lib.moe_ffn(_ptr(x), x.shape[0], _ptr(idx), _ptr(w), ctypes.byref(cw), ctypes.byref(shape), _ptr(y),
                       _ptr(ws), ws.numel(), _stream(stream)), "moe_ffn")


def decode_layer(x, Wg, weights: ExpertWeights, shape: Shape, y, ws, idx_out=None, w_out=None, flags: int = 0,
                 stream=None, cweights: Optional[_Weights] = None):
    cw = cweights if cweights is not None else weights.cstruct()
    _check(lib.moe_decode_layer(_ptr(x), x.shape[0], _ptr(Wg), ctypes.byref(cw), ctypes.byref(shape),
                                _ptr(idx_out), _ptr(w_out), _ptr(y), _ptr(ws), ws.numel(), flags,
                                _stream(stream)), "moe_decode_layer")


def decode_layer_static_scratch(x, Wg, weights: ExpertWeights, shape: Shape, y, idx_out=None, w_out=None,
                                flags: int = 0, stream=None, cweights: Optional[_Weights] = None):
    cw = cweights if cweights is not None else weights.cstruct()
    _check(lib.moe_decode_layer_static_scratch(_ptr(x), x.shape[0], _ptr(Wg), ctypes.byref(cw),
                                               ctypes.byref(shape), _ptr(idx_out), _ptr(w_out), _ptr(y), flags,
                                               _stream(stream)), "moe_decode_layer_static_scratch")


def read_status(ws, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(lib.moe_read_status(_ptr(ws), _stream(stream), ctypes.byref(v)), "moe_read_status")
    return v.value


def static_scratch_status(stream=None) -> int:
    """Device status word of this device's static scratch (synchronises)."""
    v = ctypes.c_int32(0)
    _check(lib.moe_static_scratch_status(_stream(stream), ctypes.byref(v)), "moe_static_scratch_status")
    return v.value


def mxfp4_dequant(codes, scales, K: int, out, stream=None):
    rows = codes.numel() // (K // 2)
    _check(lib.moe_mxfp4_dequant(_ptr(codes), _ptr(scales), rows, K, _ptr(out), _stream(stream)),
           "moe_mxfp4_dequant")


def set_option(option: int, value: int):
    _check(lib.moe_set_option(option, value), "moe_set_option")


def last_launch_count() -> int:
    return int(lib.moe_last_launch_count())


def lm_head(x, W, V: int, H: int, logits, ws, wfmt: int = 0, w_scale=None, flags: int = 0, stream=None):
    """logits fp32 [M, V] = x bf16 [M, H] . W^T; W bf16 [V, H] (wfmt 0) or e4m3
    codes u8 [V, H] with fp32 per-row scales w_scale [V] (wfmt 2)."""
    _check(lib.moe_lm_head(_ptr(x), x.shape[0], _ptr(W), _ptr(w_scale), V, H, wfmt, _ptr(logits), _ptr(ws),
                           ws.numel(), flags, _stream(stream)), "moe_lm_head")


def fp8_quantize(w, block: int, codes, scales, stream=None):
    rows, K = w.shape
    _check(lib.moe_fp8_quantize(_ptr(w), rows, K, block, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_fp8_quantize")


def transpose_down(w2: torch.Tensor, stream=None) -> torch.Tensor:
    """Transposed copy of down projections (moe_transpose_down): bf16
    [n, H, I] (or [H, I]) -> [n, I, H] (or [I, H]), for the split-K one-token
    layer. Weight preparation, not the hot path."""
    src = w2 if w2.dim() == 3 else w2.unsqueeze(0)
    n, H, I = src.shape
    out = torch.empty((n, I, H), dtype=w2.dtype, device=w2.device)
    _check(lib.moe_transpose_down(_ptr(src), n, H, I, _ptr(out), _stream(stream)), "moe_transpose_down")
    return out if w2.dim() == 3 else out[0]


def fp8_dequant(codes, scales, block: int, out, stream=None):
    rows, K = codes.shape
    _check(lib.moe_fp8_dequant(_ptr(codes), _ptr(scales), rows, K, block, _ptr(out), _stream(stream)),
           "moe_fp8_dequant")
