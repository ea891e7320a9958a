"""CPU oracle for the small-M MoE decode layer (Python side).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The CUDA library and its
Python binding never import this package, and this package imports nothing
from them.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp32 accumulation in
index order, or fp64); this module only marshals numpy arrays through ctypes.
Arrays of bf16 values are carried as ``numpy.uint16`` bit patterns.

Parity: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, brute force, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "moe_oracle.h")))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        # OpenMP only spreads oracle_ffn_parallel's independent expert calls
        # over threads; without it that function runs on one thread
        try:
            subprocess.check_call(cmd[:1] + ["-fopenmp"] + cmd[1:], stderr=subprocess.DEVNULL)
        except (subprocess.CalledProcessError, OSError):
            subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_mxfp4_value.argtypes = [ctypes.c_uint8, ctypes.c_uint8]
        lib.oracle_mxfp4_value.restype = ctypes.c_float
        lib.oracle_mxfp4_decode.argtypes = [P, P, i64, i32, P]
        lib.oracle_route.argtypes = [P, i32, i32, P, i32, i32, i32, P, P, P]
        lib.oracle_route_ex.argtypes = [P, i32, i32, P, i32, i32, i32, P, ctypes.c_float, i32, P, P, P]
        lib.oracle_rmsnorm.argtypes = [P, i32, i32, P, ctypes.c_float, P]
        lib.oracle_fp8_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_fp8_e4m3_value.restype = ctypes.c_double
        lib.oracle_fp8_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_fp8_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_fp8_quantize.argtypes = [P, i64, i32, i32, P, P]
        lib.oracle_lm_head.argtypes = [P, i32, i32, P, P, i32, i32, i32, P]
        lib.oracle_expert.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, i32, P]
        lib.oracle_ffn.argtypes = [P, i32, i32, P, P, i32, i32, i32, i32,
                                   P, P, P, P, P, P, i32, P, P, P, i32, P]
        lib.oracle_ffn_parallel.argtypes = [P, i32, i32, P, P, i32, i32, i32, i32,
                                            P, P, P, P, P, P, i32, P, P, P, i32, i32, P]
        lib.oracle_threads.argtypes = []
        for f in ("oracle_mxfp4_decode", "oracle_route", "oracle_expert", "oracle_ffn", "oracle_ffn_parallel",
                  "oracle_threads"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def mxfp4_value(code: int, scale: int) -> float:
    return float(_load().oracle_mxfp4_value(code & 0xFF, scale & 0xFF))


def mxfp4_decode(codes: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.size // (K // 2)
    out = np.empty((rows, K), dtype=np.float32)
    rc = _load().oracle_mxfp4_decode(_ptr(codes), _ptr(scales), rows, K, _ptr(out))
    if rc:
        raise ValueError(f"oracle_mxfp4_decode rc={rc}")
    return out


def route(x: np.ndarray, Wg: np.ndarray, k: int, acc_double: bool = False):
    """Returns (idx int32 [M,k], w float32 [M,k], logits float32 [M,E])."""
    x = _c(x, np.uint16)
    Wg = _c(Wg, np.uint16)
    M, H = x.shape
    E = Wg.shape[0]
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    logits = np.empty((M, E), dtype=np.float32)
    rc = _load().oracle_route(_ptr(x), M, H, _ptr(Wg), E, k, int(acc_double),
                              _ptr(logits), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError(f"oracle_route rc={rc}")
    return idx, w, logits


def route_ex(x: np.ndarray, Wg: np.ndarray, k: int, scoring: int = 0, bias=None, routed_scale: float = 1.0,
             acc_double: bool = False):
    """Router with scoring 0 (softmax) or 1 (sigmoid), an optional selection
    bias [E] and a routed scaling factor. Returns (idx, w, logits)."""
    x = _c(x, np.uint16)
    Wg = _c(Wg, np.uint16)
    M, H = x.shape
    E = Wg.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    logits = np.empty((M, E), dtype=np.float32)
    rc = _load().oracle_route_ex(_ptr(x), M, H, _ptr(Wg), E, k, scoring, _ptr(b), routed_scale, int(acc_double),
                                 _ptr(logits), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError(f"oracle_route_ex rc={rc}")
    return idx, w, logits


def expert(x_f32: np.ndarray, W1, W3, W2, wfmt: int = 0, S=(None, None, None),
           acc_double: bool = False) -> np.ndarray:
    """One SwiGLU expert on one token (x fp32 [H]) -> z fp32 [H]."""
    x_f32 = _c(x_f32, np.float32)
    H = x_f32.shape[0]
    dt = np.uint16 if wfmt == 0 else np.uint8
    W1, W3, W2 = _c(W1, dt), _c(W3, dt), _c(W2, dt)
    I = W1.shape[0]
    sdt = np.float32 if wfmt == 2 else np.uint8
    s1, s3, s2 = (None if s is None else _c(s, sdt) for s in S)
    z = np.empty(H, dtype=np.float32)
    rc = _load().oracle_expert(_ptr(x_f32), H, I, wfmt, _ptr(W1), _ptr(s1), _ptr(W3),
                               _ptr(s3), _ptr(W2), _ptr(s2), int(acc_double), _ptr(z))
    if rc:
        raise ValueError(f"oracle_expert rc={rc}")
    return z


def threads() -> int:
    """Host threads oracle_ffn_parallel may use (1 if built without OpenMP)."""
    return int(_load().oracle_threads())


def ffn(x: np.ndarray, idx: np.ndarray, w: np.ndarray, experts: dict, E: int, I: int,
        shared=None, wfmt: int = 0, acc_double: bool = False, nthreads: int = 1) -> np.ndarray:
    """Expert FFN with given routing.

    experts maps expert id -> (W1, W3, W2) for bf16, or
    (W1q, S1, W3q, S3, W2q, S2) for MXFP4 (u8 scales) and FP8 (fp32 scales
    per 128 elements); only the ids present in idx are
    needed. shared is (Ws1, Ws3, Ws2) bf16 or None. Returns y fp32 [M, H].
    nthreads != 1 runs the expert calls on that many host threads (0: all),
    with a bit-identical result.
    """
    x = _c(x, np.uint16)
    M, H = x.shape
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    k = idx.shape[1] if idx.ndim == 2 else 0
    keep = []  # keep contiguous copies alive during the call
    arr = {n: (ctypes.c_void_p * E)() for n in ("W1", "W3", "W2", "S1", "S3", "S2")}
    dt = np.uint16 if wfmt == 0 else np.uint8
    for e, mats in experts.items():
        if wfmt == 0:
            names = ("W1", "W3", "W2")
            vals = [_c(m, dt) for m in mats]
        else:
            names = ("W1", "S1", "W3", "S3", "W2", "S2")
            sdt = np.float32 if wfmt == 2 else np.uint8
            vals = [_c(m, np.uint8 if i % 2 == 0 else sdt) for i, m in enumerate(mats)]
        for n, v in zip(names, vals):
            keep.append(v)
            arr[n][int(e)] = v.ctypes.data
    Is = 0
    Ws = (None, None, None)
    if shared is not None:
        Ws = tuple(_c(m, np.uint16) for m in shared)
        Is = Ws[0].shape[0]
    y = np.empty((M, H), dtype=np.float32)
    if nthreads != 1:
        rc = _load().oracle_ffn_parallel(_ptr(x), M, H, _ptr(idx), _ptr(w), k, E, I, wfmt,
                                         arr["W1"], arr["S1"], arr["W3"], arr["S3"], arr["W2"], arr["S2"],
                                         Is, _ptr(Ws[0]), _ptr(Ws[1]), _ptr(Ws[2]), int(acc_double), nthreads,
                                         _ptr(y))
    else:
        rc = _load().oracle_ffn(_ptr(x), M, H, _ptr(idx), _ptr(w), k, E, I, wfmt,
                                arr["W1"], arr["S1"], arr["W3"], arr["S3"], arr["W2"], arr["S2"],
                                Is, _ptr(Ws[0]), _ptr(Ws[1]), _ptr(Ws[2]), int(acc_double), _ptr(y))
    if rc:
        raise ValueError(f"oracle_ffn rc={rc}")
    return y


def fp8_e4m3_value(code: int) -> float:
    return float(_load().oracle_fp8_e4m3_value(code & 0xFF))


def fp8_e4m3_encode(v: float) -> int:
    return int(_load().oracle_fp8_e4m3_encode(float(v)))


def fp8_quantize(w_u16: np.ndarray, block: int):
    """bf16 bits [R, K] -> (e4m3 codes u8 [R, K], fp32 scales [R, K / block])."""
    w = _c(w_u16, np.uint16)
    R, K = w.shape
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R, K // block), np.float32)
    rc = _load().oracle_fp8_quantize(_ptr(w), R, K, block, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError(f"oracle_fp8_quantize: {rc}")
    return codes, scales


def lm_head(x_u16: np.ndarray, W, V: int, wfmt: int = 0, scale=None, acc_double: bool = False) -> np.ndarray:
    """logits fp32 [M, V] of tokens x (bf16 bits [M, H]) against W (bf16 bits
    [V, H], or e4m3 codes [V, H] with fp32 per-row scale for wfmt 2)."""
    x = _c(x_u16, np.uint16)
    M, H = x.shape
    Wc = _c(W, np.uint16 if wfmt == 0 else np.uint8)
    sc = None if scale is None else _c(scale, np.float32)
    out = np.empty((M, V), np.float32)
    rc = _load().oracle_lm_head(_ptr(x), M, H, _ptr(Wc), _ptr(sc), V, wfmt, int(acc_double), _ptr(out))
    if rc:
        raise ValueError(f"oracle_lm_head: {rc}")
    return out


def rmsnorm(h_u16: np.ndarray, gamma_u16: np.ndarray, eps: float) -> np.ndarray:
    """x = bf16(h / sqrt(mean(h^2) + eps) * gamma) for bf16 bits h [M, H]."""
    h = _c(h_u16, np.uint16)
    g = _c(gamma_u16, np.uint16)
    M, H = h.shape
    x = np.empty((M, H), np.uint16)
    rc = _load().oracle_rmsnorm(_ptr(h), M, H, _ptr(g), eps, _ptr(x))
    if rc:
        raise ValueError(f"oracle_rmsnorm rc={rc}")
    return x
