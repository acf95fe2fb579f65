"""The GEMM's bounded waits, run out on purpose, without a fault: the
self-test launch withholds the first "stage ready" signal of the tiny
forward GEMM (A[256,512] . B[256,512]^T) and limits every wait to 20 ms, so
the tensor-core warp's wait gives up.  The kernel must record
MXFP4_ERR_TIMEOUT in the device status word and end cleanly, after its loads
and tensor-core operations in flight have completed.  The context stays
usable: the same GEMM then runs normally and matches the oracle, with the
status word clear."""
import time

import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu
MXFP4_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def test_withheld_signal_times_out_and_the_context_recovers(m):
    a, b = synth.tiny()
    M, K = a.shape
    N = b.shape[0]
    qa, sa = m.mxfp4_cast(a.cuda())
    qb, sb = m.mxfp4_cast(b.cuda())
    torch.cuda.synchronize()
    assert m.device_status() == 0
    c = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    m.selftest_wait_timeout(qa, sa, qb, sb, M, N, K, c, wait_limit_ms=20.0)
    torch.cuda.synchronize()  # no CUDA error: the kernel ended by itself
    elapsed = time.perf_counter() - t0
    assert m.device_status(reset=True) == MXFP4_ERR_TIMEOUT
    assert m.device_status() == 0
    assert elapsed >= 0.015  # it did wait (about the limit) before giving up

    # same operands, normal launch: correct, and the status stays clear
    y = m.gemm_fp4(qa, sa, qb, sb, M, N, K)
    torch.cuda.synchronize()
    ca, sca = oracle.cast_rows(bf16_bits(a))
    cb, scb = oracle.cast_rows(bf16_bits(b))
    ok, excess = gemm_tolerance_ok(y.float().cpu().numpy(), oracle.gemm_mxfp4(ca, sca, cb, scb, nthreads=8))
    assert ok, f"worst excess {excess:.3e}"
    assert m.device_status() == 0


def test_selftest_rejects_out_of_range_limits(m):
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    c = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    for ms in (0.5, 2500.0):  # 0.5 ms and 2.5 s: outside 1 ms .. 2 s
        with pytest.raises(m.Mxfp4Error):
            m.selftest_wait_timeout(dummy, dummy, dummy, dummy, 8, 8, 64, c, wait_limit_ms=ms)
