"""GPU parity of gemm_fp4_cast_out: the MXFP4 GEMM whose epilogue also writes
the MXFP4 casts of its own bf16 output (row-wise along N, column-wise along M).

Method: jax-aiter README, "MXFP4 training architecture" (the gradient one GEMM
produces is cast for the next one) with the "Supported ops" rows "FP4 GEMM
(low-level)" and "MXFP4 Cast".  C must be within 2^-8 |ref| + 1e-3 rms(ref)
of the fp64 oracle GEMM; the cast outputs must equal, byte for byte, the
oracle's casts of the very bf16 C the GPU wrote, scale padding (0x00)
included."""
import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def random_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    ca = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x74, 0x7C, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(0x74, 0x7C, size=(N, K // 32), dtype=np.uint8)
    return ca, sa, cb, sb


def run_cast_out(m, ca, sa, cb, sb, M, N, K, row, col, had_row, had_col):
    outs = m.gemm_fp4_cast_out(dev_u8(ca), dev_u8(oracle.sf_linear_to_tile(sa)), dev_u8(cb),
                               dev_u8(oracle.sf_linear_to_tile(sb)), M, N, K, row=row, col=col,
                               hadamard_row=had_row, hadamard_col=had_col)
    torch.cuda.synchronize()
    return outs


def check_casts(c, q_row, sf_row, q_col, sf_col, had_row, had_col):
    cbits = bf16_bits(c)
    if q_row is not None:
        codes, scales = oracle.cast_rows(cbits, hadamard=had_row)
        assert np.array_equal(q_row.cpu().numpy(), codes), "row codes"
        assert np.array_equal(sf_row.cpu().numpy(), oracle.sf_linear_to_tile(scales)), "row scales"
    if q_col is not None:
        codes, scales = oracle.cast_cols(cbits, hadamard=had_col)
        assert np.array_equal(q_col.cpu().numpy(), codes), "column codes"
        assert np.array_equal(sf_col.cpu().numpy(), oracle.sf_linear_to_tile(scales)), "column scales"


# one pair tile; M < 128 with ragged N; several tiles ragged both ways; N < 128
SHAPES = [(256, 256, 512), (96, 160, 256), (640, 544, 512), (128, 96, 64), (544, 1056, 320)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("had_row,had_col", [(False, False), (False, True), (True, True)])
def test_cast_out_parity(m, M, N, K, had_row, had_col):
    ca, sa, cb, sb = random_operands(M, N, K, seed=M * 7 + N * 3 + K + had_row + 2 * had_col)
    c, qr, sr, qc, sc = run_cast_out(m, ca, sa, cb, sb, M, N, K, True, True, had_row, had_col)
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    ok, excess = gemm_tolerance_ok(c.float().cpu().numpy(), ref)
    assert ok, f"C: worst excess over tolerance {excess:.3e}"
    check_casts(c, qr, sr, qc, sc, had_row, had_col)


@pytest.mark.parametrize("row,col", [(True, False), (False, True)])
def test_cast_out_one_output(m, row, col):
    M, N, K = 384, 288, 256
    ca, sa, cb, sb = random_operands(M, N, K, seed=11 + row)
    c, qr, sr, qc, sc = run_cast_out(m, ca, sa, cb, sb, M, N, K, row, col, False, True)
    assert (qr is None) == (not row) and (qc is None) == (not col)
    check_casts(c, qr, sr, qc, sc, False, True)


def test_cast_out_degenerate_blocks(m):
    # a zero row of A (zero blocks: scale 0x00, codes 0) and a row of A at the
    # largest scales (the products overflow fp32: non-finite blocks, 0xFF)
    M, N, K = 256, 288, 128
    ca, sa, cb, sb = random_operands(M, N, K, seed=5)
    ca[3, :] = 0
    ca[70, :] = 0x77          # every element 6.0
    sa[70, :] = 0xFE          # 2^127
    sb[:, :] = 0x90
    c, qr, sr, qc, sc = run_cast_out(m, ca, sa, cb, sb, M, N, K, True, True, False, True)
    cf = c.float().cpu().numpy()
    assert np.all(cf[3] == 0)
    check_casts(c, qr, sr, qc, sc, False, True)


@pytest.mark.parametrize("M,N,K", [(384, 288, 256), (8192, 4096, 1024)])
def test_cast_out_without_c(m, M, N, K):
    # the cast-only form (no bf16 C stored) writes the same casts as the full one
    ca, sa, cb, sb = random_operands(M, N, K, seed=M + 2 * N + K)
    full = run_cast_out(m, ca, sa, cb, sb, M, N, K, True, True, False, True)
    args = [dev_u8(ca), dev_u8(oracle.sf_linear_to_tile(sa)), dev_u8(cb), dev_u8(oracle.sf_linear_to_tile(sb))]
    c, qr, sr, qc, sc = m.gemm_fp4_cast_out(*args, M, N, K, hadamard_col=True, write_c=False)
    torch.cuda.synchronize()
    assert c is None
    for got, want in zip((qr, sr, qc, sc), full[1:]):
        assert torch.equal(got, want)
    check_casts(full[0], qr, sr, qc, sc, False, True)


def test_cast_out_k_zero_without_c(m):
    e = torch.empty(0, dtype=torch.uint8, device="cuda")
    c, qr, sr, qc, sc = m.gemm_fp4_cast_out(e, e, e, e, 96, 64, 0, hadamard_col=True, write_c=False)
    torch.cuda.synchronize()
    assert c is None
    for t in (qr, sr, qc, sc):
        assert torch.count_nonzero(t) == 0


def test_cast_out_k_zero(m):
    M, N = 64, 96
    e = torch.empty(0, dtype=torch.uint8, device="cuda")
    c, qr, sr, qc, sc = m.gemm_fp4_cast_out(e, e, e, e, M, N, 0, hadamard_col=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c) == 0
    check_casts(c, qr, sr, qc, sc, False, True)


def test_cast_out_rejects_bad_shapes(m):
    a = torch.zeros(64, 64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.Mxfp4Error):
        m.gemm_fp4_cast_out(a, s, a, s, 48, 64, 128)  # M % 32 != 0
    with pytest.raises(m.Mxfp4Error):
        m.gemm_fp4_cast_out(a, s, a, s, 64, 80, 128)  # N % 32 != 0


def test_cast_out_full_size_dgrad(m):
    # Llama-3.1-8B down projection, dgrad: dX[8192, 14336] = dY . W, with the
    # grad preset of the next cast (row plain, column Hadamard).  C must equal
    # gemm_fp4's output; the casts must equal the library's separate dual cast
    # of that C, and sampled 32-row slabs must match the oracle.
    M, N, K = 8192, 14336, 4096
    dy = synth.normal_bf16((M, K), 1e-3, seed=21).cuda()
    w = synth.normal_bf16((N, K), 0.02, seed=22).cuda()
    qa, sa = m.mxfp4_cast(dy)
    qb, sb = m.mxfp4_cast(w)
    c, qr, sr, qc, sc = m.gemm_fp4_cast_out(qa, sa, qb, sb, M, N, K, hadamard_col=True)
    c_ref = m.gemm_fp4(qa, sa, qb, sb, M, N, K)
    dual = m.mxfp4_cast_dual(c_ref, hadamard_col=True)
    torch.cuda.synchronize()
    assert torch.equal(c, c_ref)
    for got, want, what in zip((qr, sr, qc, sc), dual, ("row codes", "row scales", "col codes", "col scales")):
        assert torch.equal(got, want), what
    cb = bf16_bits(c)
    sr_np, sc_np = sr.cpu().numpy(), sc.cpu().numpy()
    qr_np, qc_np = qr.cpu().numpy(), qc.cpu().numpy()
    for r0 in (0, 4064, 8160):
        slab = cb[r0:r0 + 32]
        codes, scales = oracle.cast_rows(slab)
        assert np.array_equal(qr_np[r0:r0 + 32], codes)
        rows = np.arange(r0, r0 + 32)[:, None]
        kbs = np.arange(N // 32)[None, :]
        assert np.array_equal(sr_np[oracle.sf_tile_offset(rows, kbs, N // 32)], scales)
        codes, scales = oracle.cast_cols(slab, hadamard=True)
        assert np.array_equal(qc_np[:, r0 // 2:r0 // 2 + 16], codes)
        assert np.array_equal(sc_np[oracle.sf_tile_offset(np.arange(N), r0 // 32, M // 32)], scales[:, 0])


def test_cast_out_full_size_repeated_bit_identical(m):
    # twenty back-to-back launches of the fused dgrad of the Llama-3.1-8B down
    # projection (grad preset) into the same buffers: every byte of C and of
    # the four cast outputs equals the first launch's (the paired kernel's
    # cross-CTA hand-offs leave no room for an ordering race)
    M, N, K = 8192, 14336, 4096
    dy = synth.normal_bf16((M, K), 1e-3, seed=23).cuda()
    w = synth.normal_bf16((N, K), 0.02, seed=24).cuda()
    qa, sa = m.mxfp4_cast(dy)
    qb, sb = m.mxfp4_cast(w)
    first = m.gemm_fp4_cast_out(qa, sa, qb, sb, M, N, K, hadamard_col=True)
    ref = [t.clone() for t in first]
    for _ in range(20):
        m.gemm_fp4_cast_out(qa, sa, qb, sb, M, N, K, hadamard_col=True, c=first[0], out=first[1:])
        torch.cuda.synchronize()
        for got, want in zip(first, ref):
            assert torch.equal(got, want)
    assert m.device_status() == 0
