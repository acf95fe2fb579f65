"""Thin ctypes binding of libmxfp4.so, the GB300 (sm_103a) MXFP4 training-GEMM
library whose C ABI is declared in include/mxfp4.h.

The functions carry the C entry points' names and only marshal arguments:
torch tensors give device pointers, the current torch stream is passed as the
launch stream, and outputs not supplied by the caller are allocated with
torch.empty.  All arithmetic runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback.  If the library has not been built, every call raises.

Operations (jax-aiter README, "Supported ops" table): MXFP4 Cast (row-wise and
dual), FP4 GEMM low-level (pre-quantized operands), FP4 GEMM training
(forward, dA, dB with BF16 in/out).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libmxfp4.so")

MXFP4_OK = 0
MXFP4_ERR_CUDA = 5
MXFP4_HADAMARD_ROW = 1
MXFP4_HADAMARD_COL = 2
MXFP4_SCALE_LINEAR = 4
MXFP4_OP_FWD, MXFP4_OP_DGRAD, MXFP4_OP_WGRAD, MXFP4_OP_WGRAD_FP8 = 0, 1, 2, 3
MXFP4_GROUP_MAX = 4


class GemmDesc(ctypes.Structure):
    """mxfp4_gemm_desc: one GEMM of a gemm_fp4_grouped call."""
    _fields_ = [("a", ctypes.c_void_p), ("a_sf", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("b_sf", ctypes.c_void_p), ("c", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("ldc", ctypes.c_int64)]

class CastDesc(ctypes.Structure):
    """mxfp4_cast_desc: one cast of a mxfp4_cast_dual_grouped call."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("q_row", ctypes.c_void_p), ("sf_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("sf_col", ctypes.c_void_p), ("flags", ctypes.c_uint32)]

# Every extern "C" symbol declared in include/mxfp4.h.
ABI_SYMBOLS = (
    "mxfp4_abi_version", "mxfp4_status_string", "mxfp4_codes_bytes", "mxfp4_scales_bytes",
    "mxfp4_cast", "mxfp4_cast_dual", "gemm_fp4", "mxfp4_workspace_bytes",
    "gemm_fp4_bf16_fwd", "gemm_fp4_bf16_dgrad", "gemm_fp4_bf16_wgrad", "mxfp4_device_status",
    "gemm_fp4_bf16_fwd_noalloc", "mxfp4_last_cuda_error", "mxfp4_cuda_error_string",
    "mxfp8_cast_cols", "gemm_mxfp8", "gemm_fp8_bf16_wgrad", "gemm_fp4_cast_out",
    "mxfp4_selftest_wait_timeout", "gemm_fp4_grouped", "mxfp4_cast_dual_grouped",
)

_lib = None
_lock = threading.Lock()


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.cuda_error = 0
        msg = f"{where}: {status_string(status)} ({status})"
        if status == MXFP4_ERR_CUDA:
            self.cuda_error = lib().mxfp4_last_cuda_error()
            msg += f", CUDA error {self.cuda_error} ({lib().mxfp4_cuda_error_string(self.cuda_error).decode()})"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with quantization_mxfp4_cast_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, U32, SZ, I = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t,
                                  ctypes.c_int)
            sig = {
                "mxfp4_abi_version": (I, []),
                "mxfp4_status_string": (ctypes.c_char_p, [I]),
                "mxfp4_codes_bytes": (SZ, [I64, I64]),
                "mxfp4_scales_bytes": (SZ, [I64, I64, U32]),
                "mxfp4_cast": (I, [P, I64, I64, I64, P, P, U32, P]),
                "mxfp4_cast_dual": (I, [P, I64, I64, I64, P, P, P, P, U32, P]),
                "gemm_fp4": (I, [P, P, P, P, P, I64, I64, I64, I64, P]),
                "mxfp4_workspace_bytes": (SZ, [I, I64, I64, I64]),
                "gemm_fp4_bf16_fwd": (I, [P, P, P, I64, I64, I64, P, SZ, P]),
                "gemm_fp4_bf16_dgrad": (I, [P, P, P, I64, I64, I64, P, SZ, P]),
                "gemm_fp4_bf16_wgrad": (I, [P, P, P, I64, I64, I64, U32, P, SZ, P]),
                "mxfp4_device_status": (I, [I, ctypes.POINTER(I)]),
                "gemm_fp4_bf16_fwd_noalloc": (I, [P, P, P, I64, I64, I64, P]),
                "mxfp4_last_cuda_error": (I, []),
                "mxfp8_cast_cols": (I, [P, I64, I64, I64, P, P, U32, P]),
                "gemm_mxfp8": (I, [P, P, P, P, P, I64, I64, I64, I64, P]),
                "gemm_fp8_bf16_wgrad": (I, [P, P, P, I64, I64, I64, U32, P, SZ, P]),
                "mxfp4_cuda_error_string": (ctypes.c_char_p, [I]),
                "gemm_fp4_cast_out": (I, [P, P, P, P, P, I64, I64, I64, I64, P, P, P, P, U32, P]),
                "mxfp4_selftest_wait_timeout": (I, [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_uint64, P]),
                "gemm_fp4_grouped": (I, [ctypes.POINTER(GemmDesc), I, P]),
                "mxfp4_cast_dual_grouped": (I, [ctypes.POINTER(CastDesc), I, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mxfp4_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MXFP4_OK:
        raise Mxfp4Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def _bf16_2d(t, name):
    if t.dtype != torch.bfloat16 or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D bf16 tensor")
    if t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride")


# ----------------------------------------------------------------------------- sizes
def codes_bytes(rows: int, cols: int) -> int:
    return lib().mxfp4_codes_bytes(rows, cols)


def scales_bytes(rows: int, cols: int, linear: bool = False) -> int:
    return lib().mxfp4_scales_bytes(rows, cols, MXFP4_SCALE_LINEAR if linear else 0)


def workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return lib().mxfp4_workspace_bytes(op, M, N, K)


# ----------------------------------------------------------------------------- cast
def mxfp4_cast(x, hadamard: bool = False, linear_scales: bool = False, q=None, sf=None, stream=None):
    """Row-wise cast of bf16 x[R, C] -> (codes uint8 [R, C/2], scales uint8)."""
    _bf16_2d(x, "x")
    _need_cuda(x)
    R, C = x.shape
    if q is None:
        q = torch.empty(R, C // 2, dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(scales_bytes(R, C, linear_scales), dtype=torch.uint8, device=x.device)
    flags = (MXFP4_HADAMARD_ROW if hadamard else 0) | (MXFP4_SCALE_LINEAR if linear_scales else 0)
    _check(lib().mxfp4_cast(_ptr(x), R, C, x.stride(0), _ptr(q), _ptr(sf), flags, _stream(stream)),
           "mxfp4_cast")
    return q, sf


def mxfp4_cast_dual(x, hadamard_row: bool = False, hadamard_col: bool = False,
                    linear_scales: bool = False, out=None, stream=None):
    """Row-wise and column-wise (transposed) cast in one pass ->
    (q_row [R, C/2], sf_row, q_col [C, R/2], sf_col)."""
    _bf16_2d(x, "x")
    _need_cuda(x)
    R, C = x.shape
    if out is None:
        dev = x.device
        out = (torch.empty(R, C // 2, dtype=torch.uint8, device=dev),
               torch.empty(scales_bytes(R, C, linear_scales), dtype=torch.uint8, device=dev),
               torch.empty(C, R // 2, dtype=torch.uint8, device=dev),
               torch.empty(scales_bytes(C, R, linear_scales), dtype=torch.uint8, device=dev))
    q_row, sf_row, q_col, sf_col = out
    flags = ((MXFP4_HADAMARD_ROW if hadamard_row else 0) | (MXFP4_HADAMARD_COL if hadamard_col else 0)
             | (MXFP4_SCALE_LINEAR if linear_scales else 0))
    _check(lib().mxfp4_cast_dual(_ptr(x), R, C, x.stride(0), _ptr(q_row), _ptr(sf_row), _ptr(q_col),
                                 _ptr(sf_col), flags, _stream(stream)), "mxfp4_cast_dual")
    return q_row, sf_row, q_col, sf_col


def mxfp4_cast_dual_grouped(casts, stream=None):
    """Up to MXFP4_GROUP_MAX dual casts in one launch.  `casts` holds tuples
    (x, hadamard_row, hadamard_col[, out]); returns, per cast, the
    (q_row, sf_row, q_col, sf_col) that mxfp4_cast_dual would, byte for byte."""
    descs = (CastDesc * max(len(casts), 1))()
    outs = []
    for i, item in enumerate(casts):
        x, had_row, had_col = item[:3]
        out = item[3] if len(item) > 3 else None
        _bf16_2d(x, "x")
        _need_cuda(x)
        R, C = x.shape
        if out is None:
            dev = x.device
            out = (torch.empty(R, C // 2, dtype=torch.uint8, device=dev),
                   torch.empty(scales_bytes(R, C), dtype=torch.uint8, device=dev),
                   torch.empty(C, R // 2, dtype=torch.uint8, device=dev),
                   torch.empty(scales_bytes(C, R), dtype=torch.uint8, device=dev))
        q_row, sf_row, q_col, sf_col = out
        flags = (MXFP4_HADAMARD_ROW if had_row else 0) | (MXFP4_HADAMARD_COL if had_col else 0)
        descs[i] = CastDesc(_ptr(x), R, C, x.stride(0), _ptr(q_row), _ptr(sf_row), _ptr(q_col), _ptr(sf_col),
                            flags)
        outs.append(tuple(out))
    _check(lib().mxfp4_cast_dual_grouped(descs, len(casts), _stream(stream)), "mxfp4_cast_dual_grouped")
    return outs


# ----------------------------------------------------------------------------- GEMM
def gemm_fp4(a, a_sf, b, b_sf, M: int, N: int, K: int, c=None, stream=None):
    """C[M,N] (bf16) = A . B^T for MXFP4 operands (codes [M, K/2] / [N, K/2],
    tile-layout scales)."""
    _need_cuda(a, a_sf, b, b_sf)
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _check(lib().gemm_fp4(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K, c.stride(0),
                          _stream(stream)), "gemm_fp4")
    return c


def gemm_fp4_grouped(gemms, stream=None):
    """Independent GEMMs in one launch: `gemms` is a sequence of up to
    MXFP4_GROUP_MAX tuples (a, a_sf, b, b_sf, M, N, K) or (a, a_sf, b, b_sf,
    M, N, K, c), each as gemm_fp4's arguments.  Returns the list of C."""
    gemms = list(gemms)
    descs = (GemmDesc * max(1, len(gemms)))()
    outs = []
    for i, g in enumerate(gemms):
        a, a_sf, b, b_sf, M, N, K = g[:7]
        c = g[7] if len(g) > 7 else None
        _need_cuda(a, a_sf, b, b_sf)
        if c is None:
            c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
        descs[i] = GemmDesc(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K, c.stride(0))
        outs.append(c)
    _check(lib().gemm_fp4_grouped(descs, len(gemms), _stream(stream)), "gemm_fp4_grouped")
    return outs


def gemm_fp4_cast_out(a, a_sf, b, b_sf, M: int, N: int, K: int, row=True, col=True,
                      hadamard_row=False, hadamard_col=False, c=None, out=None, write_c=True, stream=None):
    """C[M,N] (bf16) = A . B^T like gemm_fp4, plus the MXFP4 casts of C written by
    the GEMM's epilogue: row-wise (C along N) and/or column-wise (C^T along M),
    the same bytes as mxfp4_cast_dual(C).  M, N, K multiples of 32.
    Returns (c, q_row, sf_row, q_col, sf_col); skipped outputs are None.
    `out` = (q_row, sf_row, q_col, sf_col) reuses buffers (None entries skip).
    write_c=False stores no bf16 C (c comes back None): only the casts."""
    _need_cuda(a, a_sf, b, b_sf)
    dev = a.device
    if not write_c:
        c = None
    elif c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    if out is None:
        u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)
        out = ((u8(M * N // 2).view(M, N // 2), u8(scales_bytes(M, N))) if row else (None, None)) + \
              ((u8(N * M // 2).view(N, M // 2), u8(scales_bytes(N, M))) if col else (None, None))
    q_row, sf_row, q_col, sf_col = out
    flags = (MXFP4_HADAMARD_ROW if hadamard_row else 0) | (MXFP4_HADAMARD_COL if hadamard_col else 0)
    ldc = c.stride(0) if c is not None else N
    _check(lib().gemm_fp4_cast_out(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K, ldc,
                                   _ptr(q_row), _ptr(sf_row), _ptr(q_col), _ptr(sf_col), flags,
                                   _stream(stream)),
           "gemm_fp4_cast_out")
    return c, q_row, sf_row, q_col, sf_col


def _workspace(op, M, N, K, ws, device):
    need = workspace_bytes(op, M, N, K)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return ws, ws.numel() * ws.element_size()


def gemm_fp4_bf16_fwd(x, w, y=None, ws=None, stream=None):
    """Y[M,N] = X[M,K] . W[N,K]^T through MXFP4 (both cast row-wise)."""
    _bf16_2d(x, "x"), _bf16_2d(w, "w")
    _need_cuda(x, w)
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    ws, nb = _workspace(MXFP4_OP_FWD, M, N, K, ws, x.device)
    _check(lib().gemm_fp4_bf16_fwd(_ptr(x), _ptr(w), _ptr(y), M, N, K, _ptr(ws), nb, _stream(stream)),
           "gemm_fp4_bf16_fwd")
    return y


def gemm_fp4_bf16_dgrad(dy, w, dx=None, ws=None, stream=None):
    """dX[M,K] = dY[M,N] . W[N,K] through MXFP4 (contraction over N)."""
    _bf16_2d(dy, "dy"), _bf16_2d(w, "w")
    _need_cuda(dy, w)
    M, N = dy.shape
    K = w.shape[1]
    if dx is None:
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dy.device)
    ws, nb = _workspace(MXFP4_OP_DGRAD, M, N, K, ws, dy.device)
    _check(lib().gemm_fp4_bf16_dgrad(_ptr(dy), _ptr(w), _ptr(dx), M, N, K, _ptr(ws), nb,
                                     _stream(stream)), "gemm_fp4_bf16_dgrad")
    return dx


def gemm_fp4_bf16_wgrad(dy, x, hadamard: bool = True, dw=None, ws=None, stream=None):
    """dW[N,K] = dY[M,N]^T . X[M,K] through MXFP4 (contraction over tokens M);
    with hadamard=True both operands get the 32-point transform along M."""
    _bf16_2d(dy, "dy"), _bf16_2d(x, "x")
    _need_cuda(dy, x)
    M, N = dy.shape
    K = x.shape[1]
    if dw is None:
        dw = torch.empty(N, K, dtype=torch.bfloat16, device=dy.device)
    ws, nb = _workspace(MXFP4_OP_WGRAD, M, N, K, ws, dy.device)
    flags = MXFP4_HADAMARD_COL if hadamard else 0
    _check(lib().gemm_fp4_bf16_wgrad(_ptr(dy), _ptr(x), _ptr(dw), M, N, K, flags, _ptr(ws), nb,
                                     _stream(stream)), "gemm_fp4_bf16_wgrad")
    return dw


# ----------------------------------------------------------------------------- MXFP8 (wgrad alternative)
def mxfp8_cast_cols(x, hadamard: bool = False, linear_scales: bool = False, out=None, stream=None):
    """Column-wise (transposed) MXFP8 cast of bf16 x[R, C] -> (codes uint8 [C, R]
    (E4M3, one byte per element), scales)."""
    _bf16_2d(x, "x")
    _need_cuda(x)
    R, C = x.shape
    if out is None:
        out = (torch.empty(C, R, dtype=torch.uint8, device=x.device),
               torch.empty(scales_bytes(C, R, linear_scales), dtype=torch.uint8, device=x.device))
    q, sf = out
    flags = (MXFP4_HADAMARD_COL if hadamard else 0) | (MXFP4_SCALE_LINEAR if linear_scales else 0)
    _check(lib().mxfp8_cast_cols(_ptr(x), R, C, x.stride(0), _ptr(q), _ptr(sf), flags, _stream(stream)),
           "mxfp8_cast_cols")
    return q, sf


def gemm_mxfp8(a, a_sf, b, b_sf, M: int, N: int, K: int, c=None, stream=None):
    """C[M,N] (bf16) = A . B^T for MXFP8 operands (codes [M, K] / [N, K] bytes,
    tile-layout scales)."""
    _need_cuda(a, a_sf, b, b_sf)
    if c is None:
        c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device)
    _check(lib().gemm_mxfp8(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K, c.stride(0),
                            _stream(stream)), "gemm_mxfp8")
    return c


def gemm_fp8_bf16_wgrad(dy, x, hadamard: bool = True, dw=None, ws=None, stream=None):
    """dW[N,K] = dY[M,N]^T . X[M,K] with both operands cast to MXFP8 along the
    tokens M (the FP8 alternative to gemm_fp4_bf16_wgrad)."""
    _bf16_2d(dy, "dy"), _bf16_2d(x, "x")
    _need_cuda(dy, x)
    M, N = dy.shape
    K = x.shape[1]
    if dw is None:
        dw = torch.empty(N, K, dtype=torch.bfloat16, device=dy.device)
    ws, nb = _workspace(MXFP4_OP_WGRAD_FP8, M, N, K, ws, dy.device)
    flags = MXFP4_HADAMARD_COL if hadamard else 0
    _check(lib().gemm_fp8_bf16_wgrad(_ptr(dy), _ptr(x), _ptr(dw), M, N, K, flags, _ptr(ws), nb,
                                     _stream(stream)), "gemm_fp8_bf16_wgrad")
    return dw


NOALLOC_SCRATCH_BYTES = 32 << 20  # MXFP4_NOALLOC_SCRATCH_BYTES


def gemm_fp4_bf16_fwd_noalloc(x, w, y=None, stream=None):
    """Y[M,N] = X[M,K] . W[N,K]^T like gemm_fp4_bf16_fwd, but for callers that
    cannot allocate device memory: no workspace argument, the quantized operands
    go to the library's own 32 MiB device array (shared by all calls; calls that
    overlap on the GPU race).  Sizes needing more raise Mxfp4Error
    (MXFP4_ERR_WORKSPACE).  Allocates y with torch only if it is not given."""
    _bf16_2d(x, "x"), _bf16_2d(w, "w")
    _need_cuda(x, w)
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check(lib().gemm_fp4_bf16_fwd_noalloc(_ptr(x), _ptr(w), _ptr(y), M, N, K, _stream(stream)),
           "gemm_fp4_bf16_fwd_noalloc")
    return y


def selftest_wait_timeout(a, a_sf, b, b_sf, M: int, N: int, K: int, c, wait_limit_ms: float = 20.0,
                          stream=None) -> None:
    """Run gemm_fp4's kernel with its first pipeline signal withheld and every
    wait limited to wait_limit_ms, so that a wait runs out on purpose: the
    kernel records MXFP4_ERR_TIMEOUT (read it with device_status()) and ends
    cleanly.  For tests of the failure path only; C is not a result."""
    _need_cuda(a, a_sf, b, b_sf, c)
    _check(lib().mxfp4_selftest_wait_timeout(_ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K,
                                             c.stride(0), int(wait_limit_ms * 1e6), _stream(stream)),
           "mxfp4_selftest_wait_timeout")


def device_status(reset: bool = True) -> int:
    """The library's device status word (0 = OK, 6 = a GEMM wait timed out)."""
    v = ctypes.c_int(0)
    _check(lib().mxfp4_device_status(1 if reset else 0, ctypes.byref(v)), "mxfp4_device_status")
    return v.value
