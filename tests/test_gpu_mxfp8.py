"""GPU parity of the MXFP8 (E4M3 + E8M0) wgrad alternative against the oracle:
the column-wise cast bit for bit, the kind::mxf8f6f4 GEMM and the FP8 wgrad
within |gpu - oracle| <= 2^-8 |oracle| + 1e-3 rms(oracle).

Method: jax-aiter README, "MXFP4 training architecture" (an FP8 dB path next
to the FP4 one) and "Quick start" (grad_out cast with a Hadamard transform);
format readings as stated in the oracle source."""
import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.test_oracle_mxfp8_pins import BLOCKS as E4M3_BLOCKS
from tests.test_oracle_pins import bf16_bits as golden_bits
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def check_cols(m, x, hadamard, linear):
    q, sf = m.mxfp8_cast_cols(x.cuda(), hadamard=hadamard, linear_scales=linear)
    torch.cuda.synchronize()
    R, C = x.shape
    codes, scales = oracle.cast_cols_mxfp8(bf16_bits(x), hadamard=hadamard)
    if linear:
        assert np.array_equal(sf.cpu().numpy().reshape(C, R // 32), scales), "scales differ"
    else:
        assert np.array_equal(sf.cpu().numpy(), oracle.sf_linear_to_tile(scales)), "scales differ"
    got = q.cpu().numpy()
    bad = np.argwhere(got != codes)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {tuple(bad[0])}: {got[tuple(bad[0])]:#x} vs {codes[tuple(bad[0])]:#x}"


SHAPES = [(256, 512), (128, 128), (96, 160), (32, 32), (320, 224), (640, 384)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("linear", [False, True])
def test_cast_cols_parity(m, shape, hadamard, linear):
    x = synth.normal_bf16(shape, 1.0, seed=31)
    check_cols(m, x, hadamard, linear)


def test_golden_blocks_as_columns(m):
    # each hand-worked block is one 32-row column
    cols = [golden_bits(b["x"]) for b in E4M3_BLOCKS if not b["hadamard"]]
    had_cols = [golden_bits(b["x"]) for b in E4M3_BLOCKS if b["hadamard"]]
    for group, had in ((cols, False), (had_cols, True)):
        n = len(group)
        width = ((n + 31) // 32) * 32
        bits = np.zeros((32, width), dtype=np.uint16)
        for j, c in enumerate(group):
            bits[:, j] = c
        x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        check_cols(m, x, had, linear=True)


@pytest.mark.parametrize("hadamard", [False, True])
def test_exhaustive_bf16_patterns(m, hadamard):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    arrs = [pats] + [np.random.default_rng(s).permutation(pats) for s in range(4)]
    bits = np.concatenate(arrs).reshape(256, -1)  # 256 x 1280: blocks run down the columns
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    check_cols(m, x, hadamard, linear=False)


def test_full_size_cast_config(m):
    x = synth.cast_input()  # [8192, 4096] ~ N(0,1) with 0.1% x50 outliers
    for had in (False, True):
        check_cols(m, x, had, linear=False)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (128, 256, 128), (200, 296, 320), (384, 640, 1056),
                                   (130, 264, 96), (512, 1024, 2048), (64, 512, 160), (8, 8, 32)])
def test_gemm_mxfp8_on_oracle_operands(m, M, N, K):
    a = synth.normal_bf16((M, K), 1.0, seed=41)
    b = synth.normal_bf16((N, K), 0.5, seed=42)
    ca, sa = oracle.cast_rows_mxfp8(bf16_bits(a))
    cb, sb = oracle.cast_rows_mxfp8(bf16_bits(b))
    c = m.gemm_mxfp8(to_dev(ca), to_dev(oracle.sf_linear_to_tile(sa)), to_dev(cb),
                     to_dev(oracle.sf_linear_to_tile(sb)), M, N, K)
    torch.cuda.synchronize()
    ref = oracle.gemm_mxfp8(ca, sa, cb, sb, nthreads=8)
    ok, excess = gemm_tolerance_ok(c.float().cpu().numpy(), ref)
    assert ok, f"worst excess {excess:.3e}"
    assert m.device_status() == 0


def test_gemm_mxfp8_partial_raster_group(m):
    # The kernel walks the 256-row tiles in groups sized to K (8 row tiles for
    # E4M3 at K = 8192): M = 2336 is 10 row tiles, ending in a group of 2,
    # with a ragged last row and column tile.  Random E4M3 codes (the two NaN
    # patterns replaced) and scales, against the oracle GEMM.
    M, N, K = 2336, 264, 8192
    rng = np.random.default_rng(2336)
    ca = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    ca[(ca & 0x7F) == 0x7F] = 0x3E
    cb[(cb & 0x7F) == 0x7F] = 0xBE
    sa = rng.integers(0x76, 0x7A, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(0x76, 0x7A, size=(N, K // 32), dtype=np.uint8)
    c = m.gemm_mxfp8(to_dev(ca), to_dev(oracle.sf_linear_to_tile(sa)), to_dev(cb),
                     to_dev(oracle.sf_linear_to_tile(sb)), M, N, K)
    torch.cuda.synchronize()
    ref = oracle.gemm_mxfp8(ca, sa, cb, sb, nthreads=8)
    ok, excess = gemm_tolerance_ok(c.float().cpu().numpy(), ref)
    assert ok, f"worst excess {excess:.3e}"
    assert m.device_status() == 0


@pytest.mark.parametrize("hadamard", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 384, 320), (96, 64, 128), (320, 160, 224)])
def test_fp8_wgrad(m, M, N, K, hadamard):
    dy = synth.normal_bf16((M, N), 1e-3, seed=3)
    x = synth.normal_bf16((M, K), 1.0, seed=1)
    dw = m.gemm_fp8_bf16_wgrad(dy.cuda(), x.cuda(), hadamard=hadamard)
    torch.cuda.synchronize()
    ca, sa = oracle.cast_cols_mxfp8(bf16_bits(dy), hadamard=hadamard)
    cb, sb = oracle.cast_cols_mxfp8(bf16_bits(x), hadamard=hadamard)
    ref = oracle.gemm_mxfp8(ca, sa, cb, sb, nthreads=8)
    ok, excess = gemm_tolerance_ok(dw.float().cpu().numpy(), ref)
    assert ok, f"worst excess {excess:.3e}"


@pytest.mark.slow
def test_fp8_wgrad_full_size_sampled(m):
    M, N, K, xs = synth.LLAMA_SHAPES["llama8b_down"]
    x, _, dy = synth.linear_layer(M, N, K, xs)
    dw = m.gemm_fp8_bf16_wgrad(dy.cuda(), x.cuda(), hadamard=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    sn = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 14, replace=False)]))
    sk = np.unique(np.concatenate([[0, K - 1], rng.choice(K, 46, replace=False)]))
    ca, sa = oracle.cast_cols_mxfp8(bf16_bits(dy[:, sn]), hadamard=True)
    cb, sb = oracle.cast_cols_mxfp8(bf16_bits(x[:, sk]), hadamard=True)
    ref = oracle.gemm_mxfp8(ca, sa, cb, sb, nthreads=8)
    got = dw[torch.from_numpy(sn).cuda()][:, torch.from_numpy(sk).cuda()].float().cpu().numpy()
    ok, excess = gemm_tolerance_ok(got, ref)
    assert ok, f"worst excess {excess:.3e}"
    assert m.device_status() == 0


def test_fp8_wgrad_rejects_bad_arguments(m):
    dy = torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda")  # M % 32 != 0
    x = torch.zeros(48, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.Mxfp4Error):
        m.gemm_fp8_bf16_wgrad(dy, x)
