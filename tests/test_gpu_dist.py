"""The token-sharded wgrad path of quantization_mxfp4_cast_gb300.dist on the GPU:
one NCCL rank (the only GPU), the library's casts and GEMMs, against the
oracle.  jax-aiter README, "Supported ops" row "FP4 GEMM (training)" (FSDP-aware
wgrad sharding) and "MXFP4 training architecture" (dB overlapped with the
FSDP communication).  The two-rank bookkeeping is covered on CPU
(tests/test_dist_cpu.py); here the per-shard GPU partials of two token shards
are also checked to sum to the unsharded oracle wgrad."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


@pytest.fixture(scope="module")
def mods():
    build_library()
    import quantization_mxfp4_cast_gb300 as m
    from quantization_mxfp4_cast_gb300 import dist as mdist, layer
    created = False
    if not dist.is_initialized():
        torch.cuda.set_device(0)
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{free_port()}", rank=0, world_size=1)
        created = True
    yield m, mdist, layer
    if created:
        dist.destroy_process_group()


def oracle_dx_dw(x, w, dy):
    cd, sd = oracle.cast_rows(bf16_bits(dy))
    cwc, swc = oracle.cast_cols(bf16_bits(w))
    dx = oracle.gemm_mxfp4(cd, sd, cwc, swc, nthreads=8)
    cdc, sdc = oracle.cast_cols(bf16_bits(dy), hadamard=True)
    cxc, sxc = oracle.cast_cols(bf16_bits(x), hadamard=True)
    return dx, oracle.gemm_mxfp4(cdc, sdc, cxc, sxc, nthreads=8)


def test_backward_with_overlapped_reduce_scatter(mods):
    m, mdist, L = mods
    M, N, K = 320, 256, 192
    x = synth.normal_bf16((M, K), 1.0, seed=31)
    w = synth.normal_bf16((N, K), 0.02, seed=32)
    dy = synth.normal_bf16((M, N), 1e-3, seed=33)
    x_q = L.MXFP4Quantizer.for_activation().quantize(x.cuda())
    w_q = L.MXFP4Quantizer.for_weight().quantize(w.cuda())
    dy_q = L.MXFP4Quantizer.for_grad().quantize(dy.cuda())
    dx, dw = mdist.sharded_linear_backward(dy_q, x_q, w_q)
    torch.cuda.synchronize()
    ref_dx, ref_dw = oracle_dx_dw(x, w, dy)
    assert dw.shape == (N, K)  # one rank owns every row
    for got, ref, what in ((dx, ref_dx, "dX"), (dw, ref_dw, "dW")):
        ok, excess = gemm_tolerance_ok(got.float().cpu().numpy(), ref)
        assert ok, f"{what}: worst excess {excess:.3e}"
    # one rank: the reduce-scatter is the identity, so the shard is the plain wgrad
    assert torch.equal(mdist.sharded_wgrad(dy.cuda(), x.cuda()), m.gemm_fp4_bf16_wgrad(dy.cuda(), x.cuda()))
    assert m.device_status() == 0


def test_token_shard_partials_sum_to_the_unsharded_wgrad(mods):
    # Two token shards' GPU wgrads (what two ranks compute), summed in fp32,
    # against the unsharded oracle wgrad: each partial is within the GEMM
    # tolerance of its exact value d_r, and the exact partials sum to dW.
    m, mdist, _ = mods
    M, N, K = 352, 128, 160
    x = synth.normal_bf16((M, K), 1.0, seed=34)
    dy = synth.normal_bf16((M, N), 1e-3, seed=35)
    parts, exact = [], []
    for r in range(2):
        lo, hi = mdist.shard_rows(M, 2, r)
        parts.append(m.gemm_fp4_bf16_wgrad(dy[lo:hi].cuda(), x[lo:hi].cuda()).float().cpu().numpy())
        _, d = oracle_dx_dw(x[lo:hi], torch.zeros(N, K, dtype=torch.bfloat16), dy[lo:hi])
        exact.append(d)
    _, full = oracle_dx_dw(x, torch.zeros(N, K, dtype=torch.bfloat16), dy)
    assert np.allclose(exact[0] + exact[1], full, rtol=1e-12, atol=1e-14)
    bound = sum(2.0 ** -8 * np.abs(d) + 1e-3 * np.sqrt(np.mean(d ** 2)) for d in exact)
    assert np.all(np.abs(parts[0] + parts[1] - full) <= bound)
