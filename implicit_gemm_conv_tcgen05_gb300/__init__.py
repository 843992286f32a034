"""Python binding of libigc.so, the GB300 (sm_103a) tensor-core GEMM and
implicit-GEMM convolution library.

The functions here have the names of the C ABI (include/igc.h) and do
argument marshalling only: they take torch tensors (device memory) and the
current torch CUDA stream, pass raw pointers, sizes and strides to the C
entry points, and raise IGCError on a non-zero status.  All computation runs
in the library's CUDA kernels; there is no CPU fallback.  If the library is
missing and cannot be built, importing the binding's functions raises.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
HEADER = os.path.join(_ROOT, "include", "igc.h")
DEBUG_HEADER = os.path.join(_ROOT, "include", "igc_debug.h")

IGC_OK = 0
IGC_ERR_INVALID_ARG = 1
IGC_ERR_MISALIGNED = 2
IGC_ERR_UNSUPPORTED = 3
IGC_ERR_CUDA = 4
IGC_ERR_DEVICE_TIMEOUT = 5
IGC_ERR_WORKSPACE = 6
IGC_F32 = 0
IGC_F16 = 1
IGC_BF16 = 2

_lock = threading.Lock()
_lib = None


class IGCError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    from . import build as _b
    return _b.LIB


def lib() -> ctypes.CDLL:
    """The loaded libigc.so (built in-tree on first use if out of date)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            from . import build as _b
            path = _b.build()
            if not os.path.exists(path):
                raise ImportError(f"libigc.so missing at {path}")
            L = ctypes.CDLL(path)
            i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
            L.gemm_f16.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, vp, i64, vp]
            L.gemm_f16.restype = i32
            L.gemm_bf16.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, vp, i64, vp]
            L.gemm_bf16.restype = i32
            L.gemm_s8_zp.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                     ctypes.c_int32, vp, ctypes.c_int32, vp,
                                     vp, i64, vp, i64, ctypes.c_float, vp, vp, sz, vp]
            L.gemm_s8_zp.restype = i32
            L.gemm_s8_zp_prepare.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64, vp, sz, vp]
            L.gemm_s8_zp_prepare.restype = i32
            L.gemm_s8_zp_run.argtypes = [i64, i64, i64, i32, i32, ctypes.c_int32, vp,
                                         ctypes.c_int32, vp, vp, i64, vp, i64, ctypes.c_float,
                                         vp, vp, sz, vp]
            L.gemm_s8_zp_run.restype = i32
            L.gemm_s8_zp_dequant.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                             ctypes.c_int32, vp, ctypes.c_int32, vp,
                                             vp, vp, vp, vp, i64, vp, sz, vp]
            L.gemm_s8_zp_dequant.restype = i32
            L.gemm_s8_zp_noalloc.argtypes = [i64, i64, i64, vp, i32, i64, vp, i32, i64,
                                             ctypes.c_int32, vp, ctypes.c_int32, vp,
                                             vp, i64, vp, i64, ctypes.c_float, vp, vp]
            L.gemm_s8_zp_noalloc.restype = i32
            L.gemm_s8_zp_workspace_size.argtypes = [i64, i64, i64]
            L.gemm_s8_zp_workspace_size.restype = sz
            L.conv2d_nhwc_f16_implicit.argtypes = [i32] * 11 + [vp, vp, vp, vp, vp]
            L.conv2d_nhwc_f16_implicit.restype = i32
            L.conv2d_nhwc_s8_zp.argtypes = [i32] * 11 + [vp, i32, ctypes.c_int32, vp, i32,
                                                         ctypes.c_int32, vp, vp, vp,
                                                         ctypes.c_float, vp, vp, sz, vp]
            L.conv2d_nhwc_s8_zp.restype = i32
            L.conv2d_nhwc_s8_zp_workspace_size.argtypes = [i32] * 11
            L.conv2d_nhwc_s8_zp_workspace_size.restype = sz
            L.igc_status_string.argtypes = [i32]
            L.igc_status_string.restype = ctypes.c_char_p
            L.igc_check_device_status.argtypes = [vp]
            L.igc_check_device_status.restype = i32
            L.igc_last_device_status.argtypes = []
            L.igc_last_device_status.restype = ctypes.c_uint64
            L.igc_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.igc_set_wait_limit_ns.restype = ctypes.c_uint64
            L.igc_set_tile_width.argtypes = [i32]
            L.igc_set_tile_width.restype = i32
            L.igc_set_stage_depth.argtypes = [i32]
            L.igc_set_stage_depth.restype = i32
            L.igc_set_int8_path.argtypes = [i32]
            L.igc_set_int8_path.restype = i32
            L.igc_plan_gemm.argtypes = [i32, i64, i64, i64, i32, ctypes.POINTER(ctypes.c_int32)]
            L.igc_plan_gemm.restype = i32
            L.igc_debug_wait_timeout_probe.argtypes = [vp]
            L.igc_debug_wait_timeout_probe.restype = i32
            L.igc_version.argtypes = []
            L.igc_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions a header declares (include/igc.h by default;
    include/igc_debug.h holds the tuning and test hooks)."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) -
                  {"sizeof", "defined", "if"})


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream):
    """The cudaStream_t handle (as an int) of `stream`, or of the current stream."""
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(rc: int, what: str):
    if rc != IGC_OK:
        raise IGCError(rc, what)


def _rows(t, name, dtype=None, shape=None, cuda=True):
    """(rows, cols, row stride in elements) of a 2-D row-major view; checks the
    dtype and, when given, the (rows, cols) shape, then (unless cuda is False,
    for a caller that checks devices last with _require_cuda) the device."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major view with unit inner stride")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if cuda:
        _require_cuda(**{name: t})
    return t.shape[0], t.shape[1], max(t.stride(0), t.shape[1])


def _require_cuda(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _vec(v, name, n, dtype):
    """Checks an optional per-row / per-column vector: dense, `n` elements of
    `dtype` (its device is checked by the caller's _require_cuda)."""
    if v is None:
        return
    if v.dtype != dtype or v.numel() != n or not v.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} vector of length {n}")


def _s8_outputs(C32, C8, M, N):
    """Row strides of the int8 GEMM's outputs (0 for an absent one), shapes checked."""
    import torch
    ldc32 = _rows(C32, "C32", torch.int32, (M, N), cuda=False)[2] if C32 is not None else 0
    ldc8 = _rows(C8, "C8", torch.int8, (M, N), cuda=False)[2] if C8 is not None else 0
    return ldc32, ldc8


def _s8_operands(A, Bt):
    """(M, N, K, lda, ldb) of the int8 GEMM's operands, dtypes and K checked."""
    import torch
    M, K, lda = _rows(A, "A", (torch.uint8, torch.int8), cuda=False)
    N, K2, ldb = _rows(Bt, "Bt", (torch.uint8, torch.int8), cuda=False)
    if K2 != K:
        raise ValueError("A and Bt disagree on K")
    return M, N, K, lda, ldb


def status_string(status: int) -> str:
    return lib().igc_status_string(int(status)).decode()


def igc_status_string(status: int) -> str:
    return status_string(status)


def igc_check_device_status(stream=None) -> int:
    return int(lib().igc_check_device_status(_stream(stream)))


def igc_last_device_status() -> int:
    return int(lib().igc_last_device_status())


# Tuning and test hooks (include/igc_debug.h): thread-local, they force a schedule
# choice of the calling thread's later calls only.

def igc_set_tile_width(bn: int) -> int:
    return int(lib().igc_set_tile_width(int(bn)))


def igc_set_stage_depth(k: int) -> int:
    return int(lib().igc_set_stage_depth(int(k)))


INT8_PATH_TCGEN05, INT8_PATH_MMA_SYNC, INT8_PATH_FUSED, INT8_PATH_CONVERT = 0, 1, 2, 3


def igc_set_int8_path(path: int) -> int:
    return int(lib().igc_set_int8_path(int(path)))


PLAN_GEMM_F16, PLAN_GEMM_BF16, PLAN_GEMM_S8 = 0, 1, 2
_PLAN_FIELDS = ("tile_width", "stage_k", "tiles_m", "tiles_n", "tail_start", "units", "ctas",
                "prefetch_units")


def igc_plan_gemm(op: int, M: int, N: int, K: int, clusters: int = 0) -> dict:
    """The schedule a GEMM call would run with (see include/igc.h); raises on error."""
    out = (ctypes.c_int32 * 8)()
    _check(lib().igc_plan_gemm(int(op), int(M), int(N), int(K), int(clusters), out),
           "igc_plan_gemm")
    return dict(zip(_PLAN_FIELDS, (int(v) for v in out)))


def igc_set_wait_limit_ns(limit_ns: int) -> int:
    return int(lib().igc_set_wait_limit_ns(int(limit_ns)))


def igc_debug_wait_timeout_probe(stream=None) -> int:
    return int(lib().igc_debug_wait_timeout_probe(_stream(stream)))


def igc_version() -> str:
    return lib().igc_version().decode()


# ---------------------------------------------------------------------------
# the three operations
# ---------------------------------------------------------------------------

def gemm_f16(A, Bt, C=None, C_f32_check=None, stream=None):
    """C[i,j] = sum_k A[i,k] Bt[j,k]; A (M,K) fp16, Bt (N,K) fp16 (B column-major),
    C (M,N) fp16 or fp32, C_f32_check optional fp32 (M,N).  Returns C."""
    import torch
    M, K, lda = _rows(A, "A", torch.float16)
    N, K2, ldb = _rows(Bt, "Bt", torch.float16)
    if K2 != K:
        raise ValueError("A and Bt disagree on K")
    if C is None and C_f32_check is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    c_dtype, ldc = IGC_F32, 0
    if C is not None:
        ldc = _rows(C, "C", (torch.float16, torch.float32), (M, N))[2]
        c_dtype = IGC_F16 if C.dtype == torch.float16 else IGC_F32
    ldc32 = 0
    if C_f32_check is not None:
        ldc32 = _rows(C_f32_check, "C_f32_check", torch.float32, (M, N))[2]
    rc = lib().gemm_f16(M, N, K, _ptr(A), lda, _ptr(Bt), ldb, _ptr(C), ldc, c_dtype,
                        _ptr(C_f32_check), ldc32, _stream(stream))
    _check(rc, "gemm_f16")
    return C


def gemm_bf16(A, Bt, C=None, C_f32_check=None, stream=None):
    """C[i,j] = sum_k A[i,k] Bt[j,k]; A (M,K) bf16, Bt (N,K) bf16 (B column-major),
    C (M,N) bf16 or fp32, C_f32_check optional fp32 (M,N).  Returns C."""
    import torch
    M, K, lda = _rows(A, "A", torch.bfloat16)
    N, K2, ldb = _rows(Bt, "Bt", torch.bfloat16)
    if K2 != K:
        raise ValueError("A and Bt disagree on K")
    if C is None and C_f32_check is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    c_dtype, ldc = IGC_F32, 0
    if C is not None:
        ldc = _rows(C, "C", (torch.bfloat16, torch.float32), (M, N))[2]
        c_dtype = IGC_BF16 if C.dtype == torch.bfloat16 else IGC_F32
    ldc32 = 0
    if C_f32_check is not None:
        ldc32 = _rows(C_f32_check, "C_f32_check", torch.float32, (M, N))[2]
    rc = lib().gemm_bf16(M, N, K, _ptr(A), lda, _ptr(Bt), ldb, _ptr(C), ldc, c_dtype,
                         _ptr(C_f32_check), ldc32, _stream(stream))
    _check(rc, "gemm_bf16")
    return C


def gemm_s8_zp_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().gemm_s8_zp_workspace_size(M, N, K))


def gemm_s8_zp(A, Bt, zA=0, zA_row=None, zB=0, zB_col=None, C32=None, C8=None,
               scale=0.0, scale_col=None, workspace=None, stream=None):
    """INT8 GEMM with zero points: A (M,K) uint8/int8, Bt (N,K) uint8/int8.
    Outputs C32 (M,N) int32 and/or C8 (M,N) int8.  Returns (C32, C8)."""
    import torch
    M, N, K, lda, ldb = _s8_operands(A, Bt)
    ldc32, ldc8 = _s8_outputs(C32, C8, M, N)
    _vec(zA_row, "zA_row", M, torch.int32)
    _vec(zB_col, "zB_col", N, torch.int32)
    _vec(scale_col, "scale_col", N, torch.float32)
    _require_cuda(A=A, Bt=Bt, C32=C32, C8=C8, zA_row=zA_row, zB_col=zB_col, scale_col=scale_col)
    need = gemm_s8_zp_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
    rc = lib().gemm_s8_zp(M, N, K, _ptr(A), 1 if A.dtype == torch.int8 else 0, lda,
                          _ptr(Bt), 1 if Bt.dtype == torch.int8 else 0, ldb,
                          int(zA), _ptr(zA_row), int(zB), _ptr(zB_col),
                          _ptr(C32), ldc32, _ptr(C8), ldc8, float(scale), _ptr(scale_col),
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(stream))
    _check(rc, "gemm_s8_zp")
    return C32, C8


def gemm_s8_zp_dequant(A, Bt, zA=0, zA_row=None, zB=0, zB_col=None, scale_row=None,
                       scale_col=None, bias=None, Y=None, workspace=None, stream=None):
    """INT8 GEMM with zero points and a dequantised fp32 output
    Y = ((fp32(C32) * scale_row_i) * scale_col_j) + bias_j.  Returns Y."""
    import torch
    M, N, K, lda, ldb = _s8_operands(A, Bt)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ldy = _rows(Y, "Y", torch.float32, (M, N), cuda=False)[2]
    _vec(zA_row, "zA_row", M, torch.int32)
    _vec(zB_col, "zB_col", N, torch.int32)
    _vec(scale_row, "scale_row", M, torch.float32)
    _vec(scale_col, "scale_col", N, torch.float32)
    _vec(bias, "bias", N, torch.float32)
    _require_cuda(A=A, Bt=Bt, Y=Y, zA_row=zA_row, zB_col=zB_col, scale_row=scale_row,
                  scale_col=scale_col, bias=bias)
    if workspace is None:
        workspace = torch.empty(max(gemm_s8_zp_workspace_size(M, N, K), 1), dtype=torch.uint8,
                                device=A.device)
    rc = lib().gemm_s8_zp_dequant(M, N, K, _ptr(A), 1 if A.dtype == torch.int8 else 0, lda,
                                  _ptr(Bt), 1 if Bt.dtype == torch.int8 else 0, ldb,
                                  int(zA), _ptr(zA_row), int(zB), _ptr(zB_col),
                                  _ptr(scale_row), _ptr(scale_col), _ptr(bias), _ptr(Y), ldy,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(rc, "gemm_s8_zp_dequant")
    return Y


IGC_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def gemm_s8_zp_noalloc(A, Bt, zA=0, zA_row=None, zB=0, zB_col=None, C32=None, C8=None,
                       scale=0.0, scale_col=None, stream=None):
    """gemm_s8_zp for callers that cannot allocate device memory: the library uses
    its own fixed scratch (IGC_NOALLOC_SCRATCH_BYTES per GPU) instead of a
    workspace.  Calls that overlap on the GPU race on that scratch."""
    import torch
    M, N, K, lda, ldb = _s8_operands(A, Bt)
    ldc32, ldc8 = _s8_outputs(C32, C8, M, N)
    _vec(zA_row, "zA_row", M, torch.int32)
    _vec(zB_col, "zB_col", N, torch.int32)
    _vec(scale_col, "scale_col", N, torch.float32)
    _require_cuda(A=A, Bt=Bt, C32=C32, C8=C8, zA_row=zA_row, zB_col=zB_col, scale_col=scale_col)
    rc = lib().gemm_s8_zp_noalloc(M, N, K, _ptr(A), 1 if A.dtype == torch.int8 else 0, lda,
                                  _ptr(Bt), 1 if Bt.dtype == torch.int8 else 0, ldb,
                                  int(zA), _ptr(zA_row), int(zB), _ptr(zB_col),
                                  _ptr(C32), ldc32, _ptr(C8), ldc8, float(scale), _ptr(scale_col),
                                  _stream(stream))
    _check(rc, "gemm_s8_zp_noalloc")
    return C32, C8


def gemm_s8_zp_prepare(A, Bt, workspace, M=None, N=None, K=None, stream=None):
    """Operand pre-pass of gemm_s8_zp into `workspace`; A or Bt may be None to keep
    the prepared copy of that operand (M, N, K must then be given)."""
    import torch
    lda = ldb = 0
    a_signed = b_signed = 0
    if A is not None:
        M, K, lda = _rows(A, "A", (torch.uint8, torch.int8))
        a_signed = 1 if A.dtype == torch.int8 else 0
    if Bt is not None:
        N, K2, ldb = _rows(Bt, "Bt", (torch.uint8, torch.int8))
        if K is not None and K2 != K:
            raise ValueError("A and Bt disagree on K")
        K = K2
        b_signed = 1 if Bt.dtype == torch.int8 else 0
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor")
    rc = lib().gemm_s8_zp_prepare(M, N, K, _ptr(A), a_signed, lda, _ptr(Bt), b_signed, ldb,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(rc, "gemm_s8_zp_prepare")


def gemm_s8_zp_run(M, N, K, a_signed, b_signed, workspace, zA=0, zA_row=None, zB=0, zB_col=None,
                   C32=None, C8=None, scale=0.0, scale_col=None, stream=None):
    """tcgen05 GEMM + fused zero-point correction / requantisation over a prepared workspace."""
    import torch
    M, N, K = int(M), int(N), int(K)
    ldc32, ldc8 = _s8_outputs(C32, C8, M, N)
    _vec(zA_row, "zA_row", M, torch.int32)
    _vec(zB_col, "zB_col", N, torch.int32)
    _vec(scale_col, "scale_col", N, torch.float32)
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor")
    _require_cuda(C32=C32, C8=C8, zA_row=zA_row, zB_col=zB_col, scale_col=scale_col,
                  workspace=workspace)
    rc = lib().gemm_s8_zp_run(M, N, K, int(a_signed), int(b_signed), int(zA), _ptr(zA_row),
                              int(zB), _ptr(zB_col), _ptr(C32), ldc32, _ptr(C8), ldc8,
                              float(scale), _ptr(scale_col), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gemm_s8_zp_run")
    return C32, C8


def conv2d_nhwc_f16_implicit(x, w, y=None, y_f32_check=None, pad=(1, 1), stride=(1, 1),
                             stream=None):
    """y[n,p,q,k] = sum_{r,s,c} xpad[n, p*sh+r-ph, q*sw+s-pw, c] * w[k,r,s,c];
    x NHWC fp16, w KRSC fp16, y NPQK fp16.  Returns y (or y_f32_check if y is None)."""
    import torch
    if x.dim() != 4 or w.dim() != 4 or x.dtype != torch.float16 or w.dtype != torch.float16:
        raise ValueError("x and w must be 4-D fp16 tensors")
    if not (x.is_contiguous() and w.is_contiguous() and x.is_cuda and w.is_cuda):
        raise ValueError("x and w must be dense CUDA tensors")
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    if C2 != C:
        raise ValueError("x and w disagree on C")
    ph, pw = pad
    sh, sw = stride
    P = (H + 2 * ph - R) // sh + 1
    Q = (W + 2 * pw - S) // sw + 1
    if y is None and y_f32_check is None:
        y = torch.empty((N, P, Q, K), dtype=torch.float16, device=x.device)
    for t, dt, name in ((y, torch.float16, "y"), (y_f32_check, torch.float32, "y_f32_check")):
        if t is not None and (tuple(t.shape) != (N, P, Q, K) or t.dtype != dt or not t.is_contiguous()):
            raise ValueError(f"{name} must be a dense ({N},{P},{Q},{K}) {dt} tensor")
    rc = lib().conv2d_nhwc_f16_implicit(N, H, W, C, K, R, S, ph, pw, sh, sw, _ptr(x), _ptr(w),
                                        _ptr(y), _ptr(y_f32_check), _stream(stream))
    _check(rc, "conv2d_nhwc_f16_implicit")
    return y if y is not None else y_f32_check


def conv2d_nhwc_s8_zp_workspace_size(N, H, W, C, K, R, S, pad=(1, 1), stride=(1, 1)) -> int:
    return int(lib().conv2d_nhwc_s8_zp_workspace_size(N, H, W, C, K, R, S, pad[0], pad[1],
                                                      stride[0], stride[1]))


def conv2d_nhwc_s8_zp(x, w, zX, zW=0, zW_k=None, y32=None, y8=None, scale=0.0, scale_k=None,
                      pad=(1, 1), stride=(1, 1), workspace=None, stream=None):
    """INT8 convolution with zero points (padding value zX): x NHWC uint8/int8,
    w KRSC uint8/int8; outputs y32 (int32) and/or y8 (int8), NPQK.  Returns (y32, y8)."""
    import torch
    for t, name in ((x, "x"), (w, "w")):
        if t.dim() != 4 or t.dtype not in (torch.uint8, torch.int8) or not t.is_contiguous() \
                or not t.is_cuda:
            raise ValueError(f"{name} must be a dense 4-D CUDA uint8/int8 tensor")
    N, H, W, C = x.shape
    K, R, S, C2 = w.shape
    if C2 != C:
        raise ValueError("x and w disagree on C")
    P = (H + 2 * pad[0] - R) // stride[0] + 1
    Q = (W + 2 * pad[1] - S) // stride[1] + 1
    for t, dt, name in ((y32, torch.int32, "y32"), (y8, torch.int8, "y8")):
        if t is not None and (tuple(t.shape) != (N, P, Q, K) or t.dtype != dt or not t.is_contiguous()):
            raise ValueError(f"{name} must be a dense ({N},{P},{Q},{K}) {dt} tensor")
    for v, name, dt in ((zW_k, "zW_k", torch.int32), (scale_k, "scale_k", torch.float32)):
        if v is not None and (v.dtype != dt or v.numel() != K or not v.is_contiguous() or not v.is_cuda):
            raise ValueError(f"{name} must be a contiguous CUDA {dt} vector of length {K}")
    if workspace is None:
        need = conv2d_nhwc_s8_zp_workspace_size(N, H, W, C, K, R, S, pad, stride)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    rc = lib().conv2d_nhwc_s8_zp(N, H, W, C, K, R, S, pad[0], pad[1], stride[0], stride[1],
                                 _ptr(x), 1 if x.dtype == torch.int8 else 0, int(zX),
                                 _ptr(w), 1 if w.dtype == torch.int8 else 0, int(zW), _ptr(zW_k),
                                 _ptr(y32), _ptr(y8), float(scale), _ptr(scale_k),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream))
    _check(rc, "conv2d_nhwc_s8_zp")
    return y32, y8
