"""MXFP4 oracle -- TEST INFRASTRUCTURE ONLY.

A plain CPU statement of the MXFP4 training-GEMM path (the scalar C in
``mxfp4_oracle.c`` plus fp64 NumPy glue).  Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import it; the product package never
does, and nothing here imports the product package.

Sources (page title, section):
  * jax-aiter README, "Supported ops" table, rows "MXFP4 Cast" (BF16 -> E2M1
    elements + E8M0 block scales, with a transposed copy) and "FP4 GEMM
    (low-level)" (pre-quantized fp4x2 inputs with e8m0 block scales).
  * jax-aiter README, "Supported ops" row "FP4 GEMM (training)" and
    "Quick start": FP4 forward, FP4 dA, FP4 dB with BF16 in/out; grad_out is
    cast with a Hadamard transform.
  * jax-aiter README, "MXFP4 training architecture": forward casts the
    activation row-wise and the weight both ways, then one GEMM; backward casts
    the gradient and runs the dA GEMM.

Readings where the pages are silent are stated in ``mxfp4_oracle.c``.  The
GEMM is C = A . B^T over the dequantized operands in fp64.  The layout of
scale bytes that the GEMM consumes (``sf_tile_offset``) is this library's own
boundary choice -- the pages only say the cast output is "shuffled" for the
GEMM -- and follows the public 128-row x 4-scale tile of NVIDIA's block-scaled
GEMM documentation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the scalar C oracle with gcc (no fused multiply-add)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_abi_version.restype = ctypes.c_int
            lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e2m1_magnitude_code.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_magnitude_code.restype = ctypes.c_int
            lib.oracle_block_exponent.argtypes = [ctypes.c_double]
            lib.oracle_block_exponent.restype = ctypes.c_int
            lib.oracle_fwht32_f32.argtypes = [P]
            lib.oracle_fwht32_f32.restype = None
            for name in ("oracle_cast_rows", "oracle_cast_cols"):
                f = getattr(lib, name)
                f.argtypes = [P, I64, I64, I64, ctypes.c_int, P, P]
                f.restype = ctypes.c_int
            lib.oracle_dequant_rows.argtypes = [P, P, I64, I64, P]
            lib.oracle_dequant_rows.restype = ctypes.c_int
            lib.oracle_gemm_abt_f64.argtypes = [P, P, I64, I64, I64, P, ctypes.c_int]
            lib.oracle_gemm_abt_f64.restype = ctypes.c_int
            lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_magnitude_code.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_magnitude_code.restype = ctypes.c_int
            lib.oracle_block_exponent_e4m3.argtypes = [ctypes.c_double]
            lib.oracle_block_exponent_e4m3.restype = ctypes.c_int
            for name in ("oracle_cast_rows_mxfp8", "oracle_cast_cols_mxfp8"):
                f = getattr(lib, name)
                f.argtypes = [P, I64, I64, I64, ctypes.c_int, P, P]
                f.restype = ctypes.c_int
            lib.oracle_dequant_rows_mxfp8.argtypes = [P, P, I64, I64, P]
            lib.oracle_dequant_rows_mxfp8.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def as_bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor/array (a view of the same bits)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch  # only for the bit view; no arithmetic
        return x.contiguous().view(torch.int16).numpy().view(np.uint16)
    arr = np.asarray(x)
    if arr.dtype != np.uint16:
        raise TypeError("expected bf16 bit patterns as uint16")
    return arr


# --------------------------------------------------------------------------- scalars
def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e2m1_magnitude_code(u: float) -> int:
    return _load().oracle_e2m1_magnitude_code(float(u))


def block_exponent(amax: float) -> int:
    return _load().oracle_block_exponent(float(amax))


def fwht32(y) -> np.ndarray:
    """32-point orthonormal Walsh-Hadamard transform of one block, in fp32."""
    a = np.ascontiguousarray(np.asarray(y, dtype=np.float32).copy())
    assert a.shape == (32,)
    _load().oracle_fwht32_f32(_ptr(a))
    return a


# --------------------------------------------------------------------------- cast
def cast_rows(x, hadamard: bool = False):
    """Row-wise MXFP4 cast of bf16 x[rows, cols] -> (codes [rows, cols/2] u8,
    scales [rows, cols/32] u8 in the plain linear layout)."""
    xb = np.ascontiguousarray(as_bf16_bits(x))
    rows, cols = xb.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    rc = _load().oracle_cast_rows(_ptr(xb), rows, cols, cols, int(bool(hadamard)), _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("cols must be a multiple of 32")
    return codes, scales


def cast_cols(x, hadamard: bool = False):
    """Column-wise (transposed) cast: blocks of 32 down each column of
    x[rows, cols] -> (codes [cols, rows/2], scales [cols, rows/32])."""
    xb = np.ascontiguousarray(as_bf16_bits(x))
    rows, cols = xb.shape
    codes = np.zeros((cols, rows // 2), dtype=np.uint8)
    scales = np.zeros((cols, rows // 32), dtype=np.uint8)
    rc = _load().oracle_cast_cols(_ptr(xb), rows, cols, cols, int(bool(hadamard)), _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("rows must be a multiple of 32")
    return codes, scales


def dequant_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 values of row-wise MXFP4 data (linear scales)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    out = np.empty((rows, cols), dtype=np.float64)
    rc = _load().oracle_dequant_rows(_ptr(codes), _ptr(scales), rows, cols, _ptr(out))
    if rc != 0:
        raise ValueError("bad shape")
    return out


# --------------------------------------------------------------------------- GEMM
def gemm_abt(a: np.ndarray, b: np.ndarray, nthreads: int = 1) -> np.ndarray:
    """C = A . B^T in fp64 by the straight dot-product loop (C, optionally
    split over threads by rows of C; the sums are identical either way)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    m, k = a.shape
    n, k2 = b.shape
    assert k == k2
    c = np.empty((m, n), dtype=np.float64)
    _load().oracle_gemm_abt_f64(_ptr(a), _ptr(b), m, n, k, _ptr(c), int(nthreads))
    return c


def gemm_mxfp4(codes_a, sf_a, codes_b, sf_b, nthreads: int = 1) -> np.ndarray:
    """fp64 C = dequant(A) . dequant(B)^T for row-wise MXFP4 operands with
    linear scales (A: [M, K/2] codes, [M, K/32] scales; B likewise, [N, ...])."""
    return gemm_abt(dequant_rows(codes_a, sf_a), dequant_rows(codes_b, sf_b), nthreads)


# --------------------------------------------------------------------------- MXFP8 (E4M3)
def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e4m3_magnitude_code(u: float) -> int:
    return _load().oracle_e4m3_magnitude_code(float(u))


def block_exponent_e4m3(amax: float) -> int:
    return _load().oracle_block_exponent_e4m3(float(amax))


def cast_rows_mxfp8(x, hadamard: bool = False):
    """Row-wise MXFP8 cast of bf16 x[rows, cols] -> (codes [rows, cols] u8,
    scales [rows, cols/32] u8, linear layout)."""
    xb = np.ascontiguousarray(as_bf16_bits(x))
    rows, cols = xb.shape
    codes = np.zeros((rows, cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    rc = _load().oracle_cast_rows_mxfp8(_ptr(xb), rows, cols, cols, int(bool(hadamard)), _ptr(codes),
                                        _ptr(scales))
    if rc != 0:
        raise ValueError("cols must be a multiple of 32")
    return codes, scales


def cast_cols_mxfp8(x, hadamard: bool = False):
    """Column-wise (transposed) MXFP8 cast -> (codes [cols, rows], scales [cols, rows/32])."""
    xb = np.ascontiguousarray(as_bf16_bits(x))
    rows, cols = xb.shape
    codes = np.zeros((cols, rows), dtype=np.uint8)
    scales = np.zeros((cols, rows // 32), dtype=np.uint8)
    rc = _load().oracle_cast_cols_mxfp8(_ptr(xb), rows, cols, cols, int(bool(hadamard)), _ptr(codes),
                                        _ptr(scales))
    if rc != 0:
        raise ValueError("rows must be a multiple of 32")
    return codes, scales


def dequant_rows_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, cols = codes.shape
    out = np.empty((rows, cols), dtype=np.float64)
    rc = _load().oracle_dequant_rows_mxfp8(_ptr(codes), _ptr(scales), rows, cols, _ptr(out))
    if rc != 0:
        raise ValueError("bad shape")
    return out


def gemm_mxfp8(codes_a, sf_a, codes_b, sf_b, nthreads: int = 1) -> np.ndarray:
    """fp64 C = dequant(A) . dequant(B)^T for row-wise MXFP8 operands
    (A: [M, K] codes, [M, K/32] scales; B: [N, K], [N, K/32])."""
    return gemm_abt(dequant_rows_mxfp8(codes_a, sf_a), dequant_rows_mxfp8(codes_b, sf_b), nthreads)


# --------------------------------------------------------------------------- scale tile layout
def sf_tile_offset(r, kb, kblocks: int):
    """Byte offset of the scale of row r, K-block kb inside the GEMM-ready scale
    buffer of a tensor with `kblocks` blocks per row.  Tiles of 128 rows x 4
    K-blocks (512 bytes) are stored row-tile-major, then K-tile; inside a tile
    the byte sits at (r mod 32)*16 + ((r mod 128) div 32)*4 + (kb mod 4)."""
    r = np.asarray(r, dtype=np.int64)
    kb = np.asarray(kb, dtype=np.int64)
    ktiles = (kblocks + 3) // 4
    tile = (r // 128) * ktiles + kb // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (kb % 4)


def sf_tile_bytes(rows: int, kblocks: int) -> int:
    return ((rows + 127) // 128) * ((kblocks + 3) // 4) * 512


def sf_tile_to_linear(buf: np.ndarray, rows: int, kblocks: int) -> np.ndarray:
    """Read a [rows, kblocks] linear scale array out of a tiled scale buffer."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    r, kb = np.meshgrid(np.arange(rows), np.arange(kblocks), indexing="ij")
    return buf[sf_tile_offset(r, kb, kblocks)]


def sf_linear_to_tile(lin: np.ndarray) -> np.ndarray:
    """Write a [rows, kblocks] linear scale array into a tiled buffer; padding
    bytes (rows or K-blocks past the end) are 0x00."""
    rows, kblocks = lin.shape
    out = np.zeros(sf_tile_bytes(rows, kblocks), dtype=np.uint8)
    r, kb = np.meshgrid(np.arange(rows), np.arange(kblocks), indexing="ij")
    out[sf_tile_offset(r, kb, kblocks)] = lin
    return out
