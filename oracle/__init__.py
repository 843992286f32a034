"""CPU oracle (test infrastructure only).

Plain, slow, obviously-correct C implementations of what the GPU path
computes: fp16 GEMM and direct NHWC convolution in double, int8 GEMM with zero
points in int64 plus fp32 requantisation.  See ``oracle.c`` for the
definitions and the pages they follow.

Only the tests, the package's smoke check and the benchmark's CPU-baseline /
reference arm may import this module.  It shares no code with the CUDA library
and never imports it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
          "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, no GPU needed)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
            L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f64.restype = ctypes.c_double
            L.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
            L.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
            L.oracle_f32_to_f16_rne_array.argtypes = [vp, vp, i64]
            L.oracle_f32_to_f16_rne_array.restype = None
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_f32_to_bf16_rne_array.argtypes = [vp, vp, i64]
            L.oracle_f32_to_bf16_rne_array.restype = None
            L.oracle_gemm_bf16.argtypes = [i64, i64, i64, vp, i64, vp, i64, dp, dp, i32]
            L.oracle_gemm_bf16.restype = i32
            L.oracle_dequant.argtypes = [ctypes.c_int32, vp, vp, vp]
            L.oracle_dequant.restype = ctypes.c_float
            L.oracle_dequant_matrix.argtypes = [i64, i64, vp, vp, vp, vp, vp]
            L.oracle_dequant_matrix.restype = None
            L.oracle_conv2d_nhwc_s8_zp.argtypes = [i32] * 11 + [vp, i32, ctypes.c_int32, vp, i32,
                                                                ctypes.c_int32, vp, vp, vp,
                                                                ctypes.c_float, vp, i32]
            L.oracle_conv2d_nhwc_s8_zp.restype = i32
            L.oracle_i32_to_f32_rne.argtypes = [ctypes.c_int32]
            L.oracle_i32_to_f32_rne.restype = ctypes.c_float
            L.oracle_requant.argtypes = [ctypes.c_int32, ctypes.c_float]
            L.oracle_requant.restype = ctypes.c_int8
            L.oracle_default_threads.restype = ctypes.c_int
            L.oracle_conv_out_dim.argtypes = [i32, i32, i32, i32]
            L.oracle_conv_out_dim.restype = i32
            L.oracle_gemm_f16.argtypes = [i64, i64, i64, vp, i64, vp, i64, dp, dp, i32]
            L.oracle_gemm_f16.restype = i32
            L.oracle_gemm_s8_zp.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                            ctypes.c_int32, vp, ctypes.c_int32, vp,
                                            vp, i64, vp, i64, ctypes.c_float, vp, vp, i32]
            L.oracle_gemm_s8_zp.restype = i32
            L.oracle_conv2d_nhwc_f16.argtypes = [i32] * 11 + [vp, vp, dp, dp, i32]
            L.oracle_conv2d_nhwc_f16.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(lib().oracle_default_threads())


# -------------------------------------------------------------------------
# scalar helpers
# -------------------------------------------------------------------------

def f16_to_f64(bits: int) -> float:
    return float(lib().oracle_f16_to_f64(int(bits) & 0xFFFF))


def f32_to_f16_bits(x: float) -> int:
    return int(lib().oracle_f32_to_f16_rne(float(x)))


def i32_to_f32(v: int) -> float:
    return float(lib().oracle_i32_to_f32_rne(int(v)))


def requant(c32: int, scale: float) -> int:
    return int(lib().oracle_requant(int(c32), float(scale)))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    """Round an fp32 array to fp16 (RNE) with the oracle's own conversion."""
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(flat.size, np.uint16)
    lib().oracle_f32_to_f16_rne_array(_ptr(flat), _ptr(out), flat.size)
    return out.view(np.float16).reshape(np.shape(x))


def bf16_to_f64(bits: int) -> float:
    return float(lib().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def f32_to_bf16_bits_array(x: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (RNE) with the oracle's own conversion; returns uint16 bits."""
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(flat.size, np.uint16)
    lib().oracle_f32_to_bf16_rne_array(_ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(x))


def gemm_bf16(A_bits: np.ndarray, Bt_bits: np.ndarray, nthreads: int = 0):
    """ref and sabs in double from bf16 operands given as uint16 bit arrays (M x K, N x K)."""
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    Bt = np.ascontiguousarray(Bt_bits, dtype=np.uint16)
    M, K = A.shape
    N, K2 = Bt.shape
    assert K == K2
    ref = np.empty((M, N), np.float64)
    sabs = np.empty((M, N), np.float64)
    rc = lib().oracle_gemm_bf16(M, N, K, _ptr(A), K, _ptr(Bt), K, _ptr(ref), _ptr(sabs), nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm_bf16: bad arguments")
    return ref, sabs


def dequant(c32: int, s_row=None, s_col=None, bias=None) -> float:
    """One dequantised output value; None skips a step."""
    f = lambda v: None if v is None else ctypes.byref(ctypes.c_float(v))  # noqa: E731
    return float(lib().oracle_dequant(int(c32), f(s_row), f(s_col), f(bias)))


def dequant_matrix(C32: np.ndarray, s_row=None, s_col=None, bias=None) -> np.ndarray:
    C32 = np.ascontiguousarray(C32, dtype=np.int32)
    M, N = C32.shape
    conv = lambda v: None if v is None else np.ascontiguousarray(v, dtype=np.float32)  # noqa: E731
    s_row, s_col, bias = conv(s_row), conv(s_col), conv(bias)
    Y = np.empty((M, N), np.float32)
    lib().oracle_dequant_matrix(M, N, _ptr(C32), _ptr(s_row), _ptr(s_col), _ptr(bias), _ptr(Y))
    return Y


def conv_out_dim(n: int, filt: int, pad: int, stride: int) -> int:
    return int(lib().oracle_conv_out_dim(n, filt, pad, stride))


# -------------------------------------------------------------------------
# the three operations
# -------------------------------------------------------------------------

def gemm_f16(A: np.ndarray, Bt: np.ndarray, nthreads: int = 0):
    """ref = A @ Bt.T and sabs = |A| @ |Bt|.T in double, from fp16 A (MxK), Bt (NxK)."""
    A = np.ascontiguousarray(A, dtype=np.float16)
    Bt = np.ascontiguousarray(Bt, dtype=np.float16)
    M, K = A.shape
    N, K2 = Bt.shape
    assert K == K2
    ref = np.empty((M, N), np.float64)
    sabs = np.empty((M, N), np.float64)
    rc = lib().oracle_gemm_f16(M, N, K, _ptr(A), K, _ptr(Bt), K, _ptr(ref), _ptr(sabs), nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm_f16: bad arguments")
    return ref, sabs


def gemm_s8_zp(A: np.ndarray, Bt: np.ndarray, *, a_signed: int, b_signed: int,
               zA: int = 0, zA_row=None, zB: int = 0, zB_col=None,
               scale: float = 0.0, scale_col=None, want_c8: bool = True,
               want_c64: bool = False, nthreads: int = 0):
    """Returns (C32, C8 or None, C64 or None, overflow flag)."""
    A = np.ascontiguousarray(A).view(np.uint8)
    Bt = np.ascontiguousarray(Bt).view(np.uint8)
    M, K = A.shape
    N, K2 = Bt.shape
    assert K == K2
    zA_row = None if zA_row is None else np.ascontiguousarray(zA_row, dtype=np.int32)
    zB_col = None if zB_col is None else np.ascontiguousarray(zB_col, dtype=np.int32)
    scale_col = None if scale_col is None else np.ascontiguousarray(scale_col, dtype=np.float32)
    C32 = np.empty((M, N), np.int32)
    C8 = np.empty((M, N), np.int8) if want_c8 else None
    C64 = np.empty((M, N), np.int64) if want_c64 else None
    rc = lib().oracle_gemm_s8_zp(M, N, K, _ptr(A), int(a_signed), K, _ptr(Bt), int(b_signed), K,
                                 int(zA), _ptr(zA_row), int(zB), _ptr(zB_col),
                                 _ptr(C32), N, _ptr(C8), N, float(scale), _ptr(scale_col),
                                 _ptr(C64), nthreads)
    if rc < 0:
        raise ValueError("oracle_gemm_s8_zp: bad arguments")
    return C32, C8, C64, bool(rc == 1)


def conv2d_nhwc_f16(x: np.ndarray, w: np.ndarray, pad=(1, 1), stride=(1, 1), nthreads: int = 0):
    """Direct convolution: x NHWC fp16, w KRSC fp16 -> (ref, sabs), both NPQK float64."""
    x = np.ascontiguousarray(x, dtype=np.float16)
    w = np.ascontiguousarray(w, dtype=np.float16)
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    assert C == C2
    P = conv_out_dim(H, R, pad[0], stride[0])
    Q = conv_out_dim(W, S, pad[1], stride[1])
    if P <= 0 or Q <= 0:
        raise ValueError("window does not fit")
    ref = np.empty((N, P, Q, K), np.float64)
    sabs = np.empty((N, P, Q, K), np.float64)
    rc = lib().oracle_conv2d_nhwc_f16(N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1],
                                      _ptr(x), _ptr(w), _ptr(ref), _ptr(sabs), nthreads)
    if rc != 0:
        raise ValueError("oracle_conv2d_nhwc_f16: bad arguments")
    return ref, sabs


def fp16_accept(gpu: np.ndarray, ref: np.ndarray, sabs: np.ndarray, rel: float = 2e-3):
    """Per-element acceptance |gpu - ref| <= rel * sabs; returns (ok, worst ratio)."""
    err = np.abs(gpu.astype(np.float64) - ref)
    bound = rel * sabs
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0))
    ok = bool(np.all(np.isfinite(gpu)) and np.all(err <= bound))
    return ok, float(np.max(ratio)) if ratio.size else 0.0


def conv2d_nhwc_s8_zp(x: np.ndarray, w: np.ndarray, *, x_signed: int, w_signed: int, zX: int,
                      zW: int = 0, zW_k=None, pad=(1, 1), stride=(1, 1), scale: float = 0.0,
                      scale_k=None, want_y8: bool = True, nthreads: int = 0):
    """Direct int8 convolution with zero points (padding = zX): returns (y32, y8 or None, overflow)."""
    x = np.ascontiguousarray(x).view(np.uint8)
    w = np.ascontiguousarray(w).view(np.uint8)
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    assert C == C2
    P = conv_out_dim(H, R, pad[0], stride[0])
    Q = conv_out_dim(W, S, pad[1], stride[1])
    if P <= 0 or Q <= 0:
        raise ValueError("window does not fit")
    zW_k = None if zW_k is None else np.ascontiguousarray(zW_k, dtype=np.int32)
    scale_k = None if scale_k is None else np.ascontiguousarray(scale_k, dtype=np.float32)
    y32 = np.empty((N, P, Q, K), np.int32)
    y8 = np.empty((N, P, Q, K), np.int8) if want_y8 else None
    rc = lib().oracle_conv2d_nhwc_s8_zp(N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1],
                                        _ptr(x), int(x_signed), int(zX), _ptr(w), int(w_signed),
                                        int(zW), _ptr(zW_k), _ptr(y32), _ptr(y8), float(scale),
                                        _ptr(scale_k), nthreads)
    if rc < 0:
        raise ValueError("oracle_conv2d_nhwc_s8_zp: bad arguments")
    return y32, y8, bool(rc == 1)
