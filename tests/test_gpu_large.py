"""Tensors past 2^31 elements: the dual and row-wise casts, the GEMM and the GEMM
with its output cast, at shapes whose element offsets (and byte offsets past
4 GiB) do not fit in 32 bits.  Checked against the oracle on samples that
include the last rows, the last columns and the ragged last tiles; the shapes
keep every tensor to a few GB.

Method: jax-aiter README, "Supported ops" rows "MXFP4 Cast" (CastMxfp4JA
row-wise, CastMxfp4DualJA row + transposed) and "FP4 GEMM (low-level)";
"MXFP4 training architecture" for the cast of a GEMM's own output."""
import numpy as np
import pytest
import torch

import oracle
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# 65,600 x 32,768 = 2^31 + 2^21 elements; 65,600 = 512 x 128 + 64 (a ragged last row tile)
CAST_R, CAST_C = 65600, 32768
# C[65,664, 32,768]: 2^31 + 2^22 elements, 4.3 GB of bf16; 65,664 = 256 x 256 + 128 (a half pair tile)
GEMM_M, GEMM_N, GEMM_K = 65664, 32768, 64


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


@pytest.fixture(scope="module")
def big_x():
    # N(0,1) rows, each scaled by its own power of two in [2^-20, 2^19], drawn
    # on the device (seeded) in slabs of rows
    g = torch.Generator(device="cuda").manual_seed(31)
    x = torch.empty(CAST_R, CAST_C, dtype=torch.bfloat16, device="cuda")
    step = 4096
    for r in range(0, CAST_R, step):
        n = min(step, CAST_R - r)
        e = torch.randint(-20, 20, (n, 1), device="cuda", generator=g).float()
        x[r:r + n] = (torch.randn(n, CAST_C, device="cuda", generator=g) * torch.exp2(e)).to(torch.bfloat16)
    yield x
    del x
    torch.cuda.empty_cache()


def sample_rows(n, tail, k, seed):
    # the first row, the last `tail` rows and k random ones
    rng = np.random.default_rng(seed)
    idx = np.concatenate([[0], np.arange(n - tail, n), rng.choice(n, size=k, replace=False)])
    return np.unique(idx)


def sample_cols(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=k, replace=False)]))


def gather(t, idx):
    return t[torch.from_numpy(idx).cuda()]


def check_rows(q, sf, x, rows, hadamard):
    """Row-wise codes and tile-layout scales of the sampled rows of x."""
    R, C = x.shape
    codes, scales = oracle.cast_rows(bf16_bits(gather(x, rows)), hadamard=hadamard)
    assert np.array_equal(gather(q, rows).cpu().numpy(), codes), "row codes"
    sf_h = sf.cpu().numpy()
    kb = np.arange(C // 32)
    got = sf_h[oracle.sf_tile_offset(rows[:, None], kb[None, :], C // 32)]
    assert np.array_equal(got, scales), "row scales"


def check_cols(q_col, sf_col, x, blocks, cols, hadamard):
    """Column-wise codes and scales of the sampled 32-row blocks and columns."""
    R, C = x.shape
    sf_h = sf_col.cpu().numpy()
    ci = torch.from_numpy(cols).cuda()
    q_sel = q_col[ci]
    for rb in blocks:
        xs = x[32 * rb:32 * rb + 32][:, ci]
        codes, scales = oracle.cast_cols(bf16_bits(xs), hadamard=hadamard)
        got = q_sel[:, 16 * rb:16 * rb + 16].cpu().numpy()
        assert np.array_equal(got, codes), f"column codes, row block {rb}"
        got_sf = sf_h[oracle.sf_tile_offset(cols, rb, R // 32)]
        assert np.array_equal(got_sf, scales[:, 0]), f"column scales, row block {rb}"


def test_dual_cast_past_2pow31_elements(m, big_x):
    x = big_x
    qr, sr, qc, sc = m.mxfp4_cast_dual(x, hadamard_row=True, hadamard_col=True)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    check_rows(qr, sr, x, sample_rows(CAST_R, 40, 24, seed=1), hadamard=True)
    blocks = np.unique(np.concatenate([[0, CAST_R // 32 - 2, CAST_R // 32 - 1],
                                       np.random.default_rng(2).choice(CAST_R // 32, 5, replace=False)]))
    check_cols(qc, sc, x, blocks, sample_cols(CAST_C, 62, seed=3), hadamard=True)


def test_row_cast_past_2pow31_elements(m, big_x):
    x = big_x
    q, sf = m.mxfp4_cast(x)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    check_rows(q, sf, x, sample_rows(CAST_R, 40, 24, seed=4), hadamard=False)


def random_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    ca = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x74, 0x7C, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(0x74, 0x7C, size=(N, K // 32), dtype=np.uint8)
    return ca, sa, cb, sb


def dev_operands(ca, sa, cb, sb):
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return u8(ca), u8(oracle.sf_linear_to_tile(sa)), u8(cb), u8(oracle.sf_linear_to_tile(sb))


def check_gemm_sample(c, ca, sa, cb, sb, si, sj):
    ref = oracle.gemm_mxfp4(ca[si], sa[si], cb[sj], sb[sj], nthreads=8)
    got = gather(c, si)[:, torch.from_numpy(sj).cuda()].float().cpu().numpy()
    ok, excess = gemm_tolerance_ok(got, ref)
    assert ok, f"C: worst excess over tolerance {excess:.3e}"


def test_gemm_output_past_2pow31_elements(m):
    M, N, K = GEMM_M, GEMM_N, GEMM_K
    ca, sa, cb, sb = random_operands(M, N, K, seed=41)
    c = m.gemm_fp4(*dev_operands(ca, sa, cb, sb), M, N, K)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    check_gemm_sample(c, ca, sa, cb, sb, sample_rows(M, 136, 48, seed=5), sample_cols(N, 62, seed=6))
    del c
    torch.cuda.empty_cache()


def test_gemm_output_cast_past_2pow31_elements(m):
    M, N, K = GEMM_M, GEMM_N, GEMM_K
    ca, sa, cb, sb = random_operands(M, N, K, seed=43)
    c, qr, sr, qc, sc = m.gemm_fp4_cast_out(*dev_operands(ca, sa, cb, sb), M, N, K,
                                            hadamard_col=True)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    rows = sample_rows(M, 136, 48, seed=7)
    check_gemm_sample(c, ca, sa, cb, sb, rows, sample_cols(N, 62, seed=8))
    # the casts equal the oracle's casts of the bf16 C the GPU wrote
    check_rows(qr, sr, c, rows, hadamard=False)
    blocks = np.unique(np.concatenate([[0, M // 32 - 4, M // 32 - 1],
                                       np.random.default_rng(9).choice(M // 32, 5, replace=False)]))
    check_cols(qc, sc, c, blocks, sample_cols(N, 62, seed=10), hadamard=True)
    del c, qr, sr, qc, sc
    torch.cuda.empty_cache()
