"""gemm_fp4_bf16_fwd_noalloc: the forward MXFP4 GEMM for callers that cannot
allocate device memory (a plugin whose device memory all belongs to the host
framework's allocator and that is handed only its inputs and outputs, or code
that must not make allocating CUDA calls where it runs).  It keeps its
quantized operands in the library's own fixed device array instead of a
caller workspace.

Checked here through the C ABI:
  * two calls in a row (different shapes, so the second overwrites what the
    first left in the shared array) each equal gemm_fp4_bf16_fwd bit for bit
    -- the same kernels on the same operands -- and the first also meets the
    GEMM tolerance against the oracle;
  * a call after the first takes no device memory (torch's allocator and the
    device's free bytes are unchanged);
  * the first call in a fresh process (the one that loads the array)
    returns MXFP4_OK;
  * a size that does not fit the array is refused before anything is
    launched, and bad arguments get gemm_fp4_bf16_fwd's errors.
This file sorts last so that a run stopping at the first failure has already
run every other test."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def call_noalloc(m, x, w, y):
    M, K = x.shape
    N = w.shape[0]
    return m.lib().gemm_fp4_bf16_fwd_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(y.data_ptr()),
        M, N, K, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_equals_workspace_entry_point_twice(m):
    shapes = [(512, 768, 1024, 11), (300, 1032, 2080, 12)]  # second call: ragged M, N; larger K
    cases = []
    for M, N, K, seed in shapes:
        x = synth.normal_bf16((M, K), 1.0, seed=seed)
        w = synth.normal_bf16((N, K), 0.02, seed=seed + 100)
        assert m.workspace_bytes(m.MXFP4_OP_FWD, M, N, K) <= m.NOALLOC_SCRATCH_BYTES
        xd, wd = x.cuda(), w.cuda()
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        ref = m.gemm_fp4_bf16_fwd(xd, wd)  # allocates its workspace: before the measured calls
        cases.append((x, w, xd, wd, y, ref))
    torch.cuda.synchronize()
    for i, (x, w, xd, wd, y, ref) in enumerate(cases):
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        st = call_noalloc(m, xd, wd, y)
        assert st == 0, m.status_string(st)
        torch.cuda.synchronize()
        if i > 0:  # the first call may have loaded the array; later ones take nothing
            assert torch.cuda.memory_allocated() == alloc0
            assert torch.cuda.mem_get_info()[0] >= free0
        assert torch.equal(y, ref), f"call {i}: differs from gemm_fp4_bf16_fwd"
    # the first call's result against the oracle
    x, w, _, _, y, _ = cases[0]
    ca, sa = oracle.cast_rows(bf16_bits(x))
    cb, sb = oracle.cast_rows(bf16_bits(w))
    ok, excess = gemm_tolerance_ok(y.float().cpu().numpy(), oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8))
    assert ok, f"worst excess over the tolerance {excess:.3e}"
    assert m.device_status() == 0


def test_noalloc_first_call_in_a_fresh_process():
    # the first call on a device loads the library's scratch array; in a
    # process that has made no other library call it must succeed
    code = (
        "import ctypes, torch\n"
        "import quantization_mxfp4_cast_gb300 as m\n"
        "from quantization_mxfp4_cast_gb300 import synth\n"
        "x = synth.normal_bf16((256, 512), 1.0, seed=1).cuda()\n"
        "w = synth.normal_bf16((256, 512), 0.02, seed=2).cuda()\n"
        "y = torch.empty(256, 256, dtype=torch.bfloat16, device='cuda')\n"
        "p = lambda t: ctypes.c_void_p(t.data_ptr())\n"
        "st = m.lib().gemm_fp4_bf16_fwd_noalloc(p(x), p(w), p(y), 256, 256, 512, None)\n"
        "torch.cuda.synchronize()\n"
        "print('STATUS', st, m.lib().mxfp4_last_cuda_error(), bool(torch.isfinite(y.float()).all()))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("STATUS")][-1]
    assert line == "STATUS 0 0 True", line


def test_noalloc_refuses_sizes_beyond_its_array_and_bad_arguments(m):
    M, N, K = 8192, 8192, 4096  # needs ~68 MB of quantized operands
    assert m.workspace_bytes(m.MXFP4_OP_FWD, M, N, K) > m.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, p, M, N, K, None)
    assert m.status_string(st) == "MXFP4_ERR_WORKSPACE"
    # the forward entry point's errors, in its order
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, p, 64, 64, 48, None)          # K % 32 != 0
    assert m.status_string(st) == "MXFP4_ERR_INVALID_ARG"
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, None, 0, 64, 64, None)        # M == 0: nothing to do
    assert m.status_string(st) == "MXFP4_OK"
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, None, 64, 64, 64, None)       # no output
    assert m.status_string(st) == "MXFP4_ERR_INVALID_ARG"
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, p, 64, 60, 64, None)          # N % 8 != 0
    assert m.status_string(st) == "MXFP4_ERR_MISALIGNED"
    st = m.lib().gemm_fp4_bf16_fwd_noalloc(p, p, p, 8192, 8192, 4016, None)   # bad K before the size
    assert m.status_string(st) == "MXFP4_ERR_INVALID_ARG"
