"""gemm_fp4_bf16_fwd_noalloc: the forward MXFP4 GEMM for callers that cannot
allocate device memory (code that may not make allocating CUDA calls, or a
plugin that owns no device memory beyond its inputs and outputs).  It keeps
its quantized operands in the library's own fixed device array instead of a
caller workspace.

Checked here through the C ABI: two calls in a row (different shapes, so the
second overwrites what the first left in the shared array) each agree with
gemm_fp4_bf16_fwd within the GEMM tolerance used by the other tests, and a
size that does not fit the array is refused before anything is launched.
This file sorts last so that a run stopping at the first failure has already
run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from quantization_mxfp4_cast_gb300 import synth
from tests.util import build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def call_noalloc(m, x, w):
    M, K = x.shape
    N = w.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=x.device)
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(y.data_ptr()),
        M, N, K, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, y


def test_noalloc_matches_workspace_entry_point_twice(m):
    shapes = [(512, 768, 1024, 11), (300, 1032, 2080, 12)]  # second call: ragged M, N; larger K
    for M, N, K, seed in shapes:
        x = synth.normal_bf16((M, K), 1.0, seed=seed).cuda()
        w = synth.normal_bf16((N, K), 0.02, seed=seed + 100).cuda()
        assert m.workspace_bytes(m.MXFP4_OP_FWD, M, N, K) <= m.NOALLOC_SCRATCH_BYTES
        st, y = call_noalloc(m, x, w)
        assert st == 0, m.status_string(st)
        ref = m.gemm_fp4_bf16_fwd(x, w)
        torch.cuda.synchronize()
        ok, excess = gemm_tolerance_ok(y.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64))
        assert ok, f"{M}x{N}x{K}: worst excess {excess:.3e}"
    assert m.device_status() == 0


def test_noalloc_refuses_sizes_beyond_its_array(m):
    M, N, K = 8192, 8192, 4096  # needs ~68 MB of quantized operands
    assert m.workspace_bytes(m.MXFP4_OP_FWD, M, N, K) > m.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, p, M, N, K, None)
    assert m.status_string(st) == "MXFP4_ERR_WORKSPACE"
