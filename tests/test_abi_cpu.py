"""CPU checks of the C ABI: the library builds, loads and exports every symbol
include/mxfp4.h declares; size queries and host-side argument validation.
Every call here returns before the library touches CUDA (no compute without a
GPU)."""
import ctypes
import os
import re

import pytest

from tests.util import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_library()
    import quantization_mxfp4_cast_gb300 as m
    return m.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return names


def test_header_declares_the_abi():
    import quantization_mxfp4_cast_gb300 as m
    names = declared_functions()
    assert sorted(names) == sorted(m.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.mxfp4_abi_version() == 1


def test_status_strings(L):
    import quantization_mxfp4_cast_gb300 as m
    for s, name in enumerate(["MXFP4_OK", "MXFP4_ERR_INVALID_ARG", "MXFP4_ERR_MISALIGNED",
                              "MXFP4_ERR_UNSUPPORTED_DEVICE", "MXFP4_ERR_WORKSPACE", "MXFP4_ERR_CUDA",
                              "MXFP4_ERR_TIMEOUT", "MXFP4_ERR_NOT_IMPLEMENTED"]):
        assert m.status_string(s) == name
    assert m.status_string(99) == "MXFP4_UNKNOWN_STATUS"


def test_size_queries_match_the_oracle_layout(L):
    import oracle
    import quantization_mxfp4_cast_gb300 as m
    for rows, cols in [(1, 32), (128, 128), (129, 160), (8192, 4096), (300, 96)]:
        assert m.codes_bytes(rows, cols) == rows * cols // 2
        assert m.scales_bytes(rows, cols, linear=True) == rows * cols // 32
        assert m.scales_bytes(rows, cols) == oracle.sf_tile_bytes(rows, cols // 32)
    M, N, K = 300, 520, 1056

    def carve(r, c):
        a = lambda n: (n + 255) // 256 * 256
        return a(r * c // 2) + a(oracle.sf_tile_bytes(r, c // 32))
    assert m.workspace_bytes(m.MXFP4_OP_FWD, M, N, K) == carve(M, K) + carve(N, K)
    assert m.workspace_bytes(m.MXFP4_OP_DGRAD, M, N, K) == carve(M, N) + carve(K, N)
    assert m.workspace_bytes(m.MXFP4_OP_WGRAD, M, N, K) == carve(N, M) + carve(K, M)
    assert m.workspace_bytes(7, M, N, K) == 0


def test_argument_validation_before_any_launch(L):
    P = ctypes.c_void_p
    good = P(0x10000)      # never dereferenced: validation fails first
    odd = P(0x10008)
    INV, MIS, WS = 1, 2, 4
    # cols not a multiple of 32
    assert L.mxfp4_cast(good, 4, 48, 48, good, good, 0, None) == INV
    # unknown flag bits
    assert L.mxfp4_cast(good, 4, 64, 64, good, good, 8, None) == INV
    assert L.mxfp4_cast(good, 4, 64, 64, good, good, 2, None) == INV  # column transform on a row cast
    # null input / outputs
    assert L.mxfp4_cast(None, 4, 64, 64, good, good, 0, None) == INV
    assert L.mxfp4_cast(good, 4, 64, 64, None, good, 0, None) == INV
    # misaligned input pointer or pitch
    assert L.mxfp4_cast(odd, 4, 64, 64, good, good, 0, None) == MIS
    assert L.mxfp4_cast(good, 4, 64, 68, good, good, 0, None) == MIS
    # pitch smaller than a row
    assert L.mxfp4_cast(good, 4, 64, 32, good, good, 0, None) == INV
    # dual cast needs rows % 32 == 0
    assert L.mxfp4_cast_dual(good, 48, 64, 64, good, good, good, good, 0, None) == INV
    # empty inputs are a no-op
    assert L.mxfp4_cast(None, 0, 64, 64, None, None, 0, None) == 0
    assert L.mxfp4_cast_dual(None, 0, 64, 64, None, None, None, None, 0, None) == 0
    # GEMM: K % 32, ldc < N, misaligned ldc, negative sizes, empty output
    assert L.gemm_fp4(good, good, good, good, good, 8, 8, 48, 8, None) == INV
    assert L.gemm_fp4(good, good, good, good, good, 8, 16, 64, 8, None) == INV
    assert L.gemm_fp4(good, good, good, good, good, 8, 12, 64, 12, None) == MIS
    assert L.gemm_fp4(good, good, good, good, good, -1, 8, 64, 8, None) == INV
    assert L.gemm_fp4(None, None, None, None, None, 0, 8, 64, 8, None) == 0
    # bf16 entry points: missing / short workspace
    assert L.gemm_fp4_bf16_fwd(good, good, good, 64, 64, 64, None, 0, None) == WS
    assert L.gemm_fp4_bf16_fwd(good, good, good, 64, 64, 64, good, 16, None) == WS
    assert L.gemm_fp4_bf16_dgrad(good, good, good, 64, 48, 64, good, 1 << 30, None) == INV
    assert L.gemm_fp4_bf16_wgrad(good, good, good, 48, 64, 64, 0, good, 1 << 30, None) == INV
    assert L.gemm_fp4_bf16_wgrad(good, good, good, 64, 64, 64, 1, good, 1 << 30, None) == INV
    # GEMM with the output cast: M and N multiples of 32, tile-layout flags
    # only, codes and scales given together, aligned outputs, empty no-op
    co = L.gemm_fp4_cast_out
    assert co(good, good, good, good, good, 48, 64, 64, 64, good, good, good, good, 0, None) == INV
    assert co(good, good, good, good, good, 64, 48, 64, 48, good, good, good, good, 0, None) == INV
    assert co(good, good, good, good, good, 64, 64, 64, 64, good, good, good, good, 4, None) == INV
    assert co(good, good, good, good, good, 64, 64, 64, 64, good, None, good, good, 0, None) == INV
    assert co(good, good, good, good, good, 64, 64, 64, 64, good, good, odd, good, 0, None) == MIS
    assert co(None, None, None, None, None, 0, 64, 64, 64, None, None, None, None, 2, None) == 0
    # no output at all (no C and no cast) is refused; no C with a cast output is fine to validate
    assert co(good, good, good, good, None, 64, 64, 64, 64, None, None, None, None, 0, None) == INV
    assert co(good, good, good, good, None, 64, 64, 64, 0, good, good, odd, good, 0, None) == MIS
    # grouped GEMM: count 1..4, a non-null array, each descriptor checked as
    # gemm_fp4 checks its arguments (the first failing one's status), empty
    # descriptors skipped
    from quantization_mxfp4_cast_gb300 import GemmDesc
    D = lambda M, N, K, ldc, c=good, a=good: GemmDesc(a, good, good, good, c, M, N, K, ldc)
    grp = lambda *ds: L.gemm_fp4_grouped((GemmDesc * len(ds))(*ds), len(ds), None)
    assert L.gemm_fp4_grouped(None, 1, None) == INV
    assert L.gemm_fp4_grouped((GemmDesc * 1)(D(0, 8, 64, 8)), 0, None) == INV
    assert L.gemm_fp4_grouped((GemmDesc * 5)(*[D(0, 8, 64, 8)] * 5), 5, None) == INV
    assert grp(D(8, 8, 48, 8)) == INV                       # K % 32
    assert grp(D(0, 8, 64, 8), D(8, 12, 64, 12)) == MIS     # second descriptor: ldc % 8
    assert grp(D(8, 8, 64, 8, a=odd)) == MIS                 # misaligned operand
    assert grp(D(8, 8, 64, 8, c=None)) == INV                # missing output
    assert grp(D(0, 8, 64, 8, c=None), D(8, 0, 64, 8, c=None)) == 0   # all empty: no-op
    # grouped dual cast: the same rules, each descriptor checked as
    # mxfp4_cast_dual checks its arguments
    from quantization_mxfp4_cast_gb300 import CastDesc
    C = lambda R, Cc, ldx, x=good, q=good, fl=0: CastDesc(x, R, Cc, ldx, q, good, good, good, fl)
    cgrp = lambda *ds: L.mxfp4_cast_dual_grouped((CastDesc * len(ds))(*ds), len(ds), None)
    assert L.mxfp4_cast_dual_grouped(None, 1, None) == INV
    assert L.mxfp4_cast_dual_grouped((CastDesc * 1)(C(0, 64, 64)), 0, None) == INV
    assert L.mxfp4_cast_dual_grouped((CastDesc * 5)(*[C(0, 64, 64)] * 5), 5, None) == INV
    assert cgrp(C(48, 64, 64)) == INV                        # rows % 32
    assert cgrp(C(0, 64, 64), C(32, 48, 64)) == INV          # second descriptor: cols % 32
    assert cgrp(C(32, 64, 64, x=odd)) == MIS                 # misaligned input
    assert cgrp(C(32, 64, 64, q=None)) == INV                # missing output
    assert cgrp(C(32, 64, 64, fl=8)) == INV                  # unknown flag
    assert cgrp(C(0, 64, 64, x=None), C(32, 0, 64, x=None)) == 0   # all empty: no-op
    st = ctypes.c_int(0)
    assert L.mxfp4_device_status(0, None) == INV


def test_cuda_error_diagnostic(L):
    assert L.mxfp4_last_cuda_error() == 0          # no CUDA failure in this thread yet
    assert L.mxfp4_cuda_error_string(0) == b"cudaSuccess"
