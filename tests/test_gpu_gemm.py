"""GPU parity of the block-scaled MXFP4 GEMM (tcgen05 kind::mxf4) against the
fp64 oracle: |gpu - oracle| <= 2^-8 |oracle| + 1e-3 rms(oracle) elementwise.

Method: jax-aiter README, "Supported ops" rows "FP4 GEMM (low-level)"
(gemm_fp4 on pre-quantized fp4x2 + e8m0 operands) and "FP4 GEMM (training)"
(A[M,K] . B[N,K]^T, BF16 in/out, FP4 forward, dA and dB; grad_out cast with a
Hadamard transform)."""
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


def to_dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gemm_fp4(m, ca, sa, cb, sb, M, N, K):
    c = m.gemm_fp4(to_dev_u8(ca), to_dev_u8(oracle.sf_linear_to_tile(sa)), to_dev_u8(cb),
                   to_dev_u8(oracle.sf_linear_to_tile(sb)), M, N, K)
    torch.cuda.synchronize()
    return c.float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, what=""):
    ok, excess = gemm_tolerance_ok(gpu, ref)
    assert ok, f"{what}: worst excess over tolerance {excess:.3e}"


GEMM_SHAPES = [(256, 256, 512), (128, 256, 256), (200, 296, 320), (1, 8, 32), (384, 640, 1056),
               (130, 264, 96), (512, 1024, 2048), (64, 512, 160)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_fp4_on_oracle_operands(m, M, N, K):
    xa = synth.with_outliers(synth.normal_bf16((M, K), 1.0, seed=M + K), frac=0.01)
    xb = synth.normal_bf16((N, K), 0.02, seed=N + 3 * K)
    ca, sa = oracle.cast_rows(bf16_bits(xa))
    cb, sb = oracle.cast_rows(bf16_bits(xb))
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(run_gemm_fp4(m, ca, sa, cb, sb, M, N, K), ref, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (160, 136, 384)])
def test_gemm_fp4_random_codes_and_scales(m, M, N, K):
    # every code value and a spread of scales, independent of the cast
    rng = np.random.default_rng(M * N + K)
    ca = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x70, 0x8F, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(0x70, 0x8F, size=(N, K // 32), dtype=np.uint8)
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(run_gemm_fp4(m, ca, sa, cb, sb, M, N, K), ref)


@pytest.mark.parametrize("M,N,K", [(2336, 520, 14336), (8488, 264, 4096)])
def test_gemm_fp4_partial_raster_group(m, M, N, K):
    # The kernel walks the 256-row tiles in groups sized to K (8 row tiles at
    # K = 14336, 32 at K = 4096); these shapes end in a partial group (10 =
    # 8 + 2 and 34 = 32 + 2 row tiles) with a ragged last row and column tile.
    rng = np.random.default_rng(M + N + K)
    ca = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x76, 0x7A, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(0x76, 0x7A, size=(N, K // 32), dtype=np.uint8)
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(run_gemm_fp4(m, ca, sa, cb, sb, M, N, K), ref, f"{M}x{N}x{K}")


def test_gemm_fp4_one_hot_scales(m):
    # all codes 1.0; one scale byte raised per operand: isolates the scale
    # addressing (row, block) of both operands exactly
    M, N, K = 256, 512, 512
    ca = np.full((M, K // 2), 0x22, dtype=np.uint8)
    cb = np.full((N, K // 2), 0x22, dtype=np.uint8)
    for (ra, ka, rb, kb) in [(0, 0, 0, 0), (37, 5, 300, 11), (200, 15, 511, 3), (129, 8, 130, 9)]:
        sa = np.full((M, K // 32), 0x7F, dtype=np.uint8)
        sb = np.full((N, K // 32), 0x7F, dtype=np.uint8)
        sa[ra, ka] = 0x81
        sb[rb, kb] = 0x80
        ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
        got = run_gemm_fp4(m, ca, sa, cb, sb, M, N, K)
        assert np.array_equal(got, ref), (ra, ka, rb, kb)


def test_tiny_forward_config(m):
    a, b = synth.tiny()
    y = m.gemm_fp4_bf16_fwd(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    ca, sa = oracle.cast_rows(bf16_bits(a))
    cb, sb = oracle.cast_rows(bf16_bits(b))
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(y.float().cpu().numpy(), ref, "tiny fwd")


@pytest.mark.parametrize("M,N,K", [(256, 384, 320), (96, 64, 128), (320, 160, 224)])
def test_dgrad(m, M, N, K):
    dy = synth.normal_bf16((M, N), 1e-3, seed=3)
    w = synth.normal_bf16((N, K), 0.02, seed=2)
    dx = m.gemm_fp4_bf16_dgrad(dy.cuda(), w.cuda())
    torch.cuda.synchronize()
    ca, sa = oracle.cast_rows(bf16_bits(dy))
    cb, sb = oracle.cast_cols(bf16_bits(w))
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(dx.float().cpu().numpy(), ref, "dgrad")


@pytest.mark.parametrize("hadamard", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 384, 320), (96, 64, 128), (320, 160, 224)])
def test_wgrad(m, M, N, K, hadamard):
    dy = synth.normal_bf16((M, N), 1e-3, seed=3)
    x = synth.normal_bf16((M, K), 1.0, seed=1)
    dw = m.gemm_fp4_bf16_wgrad(dy.cuda(), x.cuda(), hadamard=hadamard)
    torch.cuda.synchronize()
    ca, sa = oracle.cast_cols(bf16_bits(dy), hadamard=hadamard)
    cb, sb = oracle.cast_cols(bf16_bits(x), hadamard=hadamard)
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    assert_close(dw.float().cpu().numpy(), ref, "wgrad")


def test_k_zero_and_empty(m):
    c = torch.full((8, 16), 7.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    m.gemm_fp4(dummy, dummy, dummy, dummy, 8, 16, 0, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)
    e = torch.empty(0, 16, dtype=torch.bfloat16, device="cuda")
    m.gemm_fp4(dummy, dummy, dummy, dummy, 0, 16, 64, c=e)


def test_deterministic_and_side_stream(m):
    M, N, K = 1024, 2048, 4096
    x = synth.normal_bf16((M, K), 1.0, seed=1)
    w = synth.normal_bf16((N, K), 0.02, seed=2)
    y0 = m.gemm_fp4_bf16_fwd(x.cuda(), w.cuda())
    s = torch.cuda.Stream()
    ballast = torch.randn(8192, 8192, device="cuda")
    xd = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        for _ in range(4):
            ballast = ballast @ ballast * 1e-4
        xd.copy_(x.cuda())
        y1 = m.gemm_fp4_bf16_fwd(xd, w.cuda(), stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert m.device_status() == 0


def sample_idx(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = rng.choice(n, size=min(k, n), replace=False)
    idx[:2] = [0, n - 1] if n > 1 else [0, 0]
    return np.unique(idx)


# Full-size outputs are checked on a 64 x 64 sample spread over C: 4096 oracle
# values, over which the tolerance's rms is taken.
N_SAMPLE = 64


def check_sampled_fwd(m, x, w, y, seed):
    M, K = x.shape
    N = w.shape[0]
    si, sj = sample_idx(M, N_SAMPLE, seed), sample_idx(N, N_SAMPLE, seed + 1)
    ca, sa = oracle.cast_rows(bf16_bits(x[si]))
    cb, sb = oracle.cast_rows(bf16_bits(w[sj]))
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    got = y[torch.from_numpy(si).cuda()][:, torch.from_numpy(sj).cuda()].float().cpu().numpy()
    assert_close(got, ref, "sampled fwd")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama8b_gate_up"])
def test_full_size_forward_sampled(m, name):
    M, N, K, xs = synth.LLAMA_SHAPES[name]
    x, w, _ = synth.linear_layer(M, N, K, xs)
    y = m.gemm_fp4_bf16_fwd(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    check_sampled_fwd(m, x, w, y, seed=5)
    assert m.device_status() == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama8b_down", "llama70b_qkv", "llama70b_o", "llama70b_gate_up",
                                  "llama70b_down"])
def test_full_size_train_step_sampled(m, name):
    # fwd Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X (Hadamard along the tokens)
    # on a Llama layer: e.g. 8B down projection X[8192,14336], W[4096,14336], dY[8192,4096]
    M, N, K, xs = synth.LLAMA_SHAPES[name]
    x, w, dy = synth.linear_layer(M, N, K, xs)
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    y = m.gemm_fp4_bf16_fwd(xd, wd)
    dx = m.gemm_fp4_bf16_dgrad(dyd, wd)
    dw = m.gemm_fp4_bf16_wgrad(dyd, xd, hadamard=True)
    torch.cuda.synchronize()
    check_sampled_fwd(m, x, w, y, seed=6)
    si, sk = sample_idx(M, N_SAMPLE, 7), sample_idx(K, N_SAMPLE, 8)
    ca, sa = oracle.cast_rows(bf16_bits(dy[si]))
    cb, sb = oracle.cast_cols(bf16_bits(w[:, sk]))
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    got = dx[torch.from_numpy(si).cuda()][:, torch.from_numpy(sk).cuda()].float().cpu().numpy()
    assert_close(got, ref, "sampled dgrad")
    sn, sk = sample_idx(N, N_SAMPLE, 9), sample_idx(K, N_SAMPLE, 10)
    ca, sa = oracle.cast_cols(bf16_bits(dy[:, sn]), hadamard=True)
    cb, sb = oracle.cast_cols(bf16_bits(x[:, sk]), hadamard=True)
    ref = oracle.gemm_mxfp4(ca, sa, cb, sb, nthreads=8)
    got = dw[torch.from_numpy(sn).cuda()][:, torch.from_numpy(sk).cuda()].float().cpu().numpy()
    assert_close(got, ref, "sampled wgrad")
    assert m.device_status() == 0


@pytest.mark.slow
def test_repeated_full_size_dgrad_is_bit_identical(m):
    # The CTA pair hands stages and the accumulator between its two SMs through
    # mbarriers with CTA-scope release; a rare ordering race would show as a
    # launch whose output differs.  24 back-to-back launches of the 8B
    # down-projection dgrad (dX[8192,14336] = dY . W, 1792 tiles each) must all
    # equal the first, bit for bit.
    M, N, K, xs = synth.LLAMA_SHAPES["llama8b_down"]
    _, w, dy = synth.linear_layer(M, N, K, xs)
    qdy = m.mxfp4_cast_dual(dy.cuda())
    qw = m.mxfp4_cast_dual(w.cuda())
    outs = [torch.empty(M, K, dtype=torch.bfloat16, device="cuda") for _ in range(24)]
    for c in outs:
        m.gemm_fp4(qdy[0], qdy[1], qw[2], qw[3], M, K, N, c=c)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    for i, c in enumerate(outs[1:], 1):
        assert torch.equal(c, outs[0]), f"launch {i} differs from launch 0"
    assert torch.isfinite(outs[0].float()).all()


def rand_operands(M, N, K, seed, dev="cuda"):
    """Random codes and tile-layout scales (every code value, a spread of
    power-of-two scales) for a gemm_fp4 call, generated on the device."""
    import quantization_mxfp4_cast_gb300 as mod
    g = torch.Generator(device=dev).manual_seed(seed)
    u8 = lambda *shape, lo=0, hi=256: torch.randint(lo, hi, shape, dtype=torch.uint8, device=dev, generator=g)
    return (u8(M, K // 2), u8(mod.scales_bytes(M, K), lo=0x76, hi=0x7A),
            u8(N, K // 2), u8(mod.scales_bytes(N, K), lo=0x76, hi=0x7A))


def test_grouped_gemm_is_bit_identical_to_separate_calls(m):
    # One launch over the train step's three GEMMs of the 8B down projection
    # (fwd 8192x4096x14336, dgrad 8192x14336x4096, wgrad 4096x14336x8192) and
    # a ragged one with a K tail (K % 64 == 32): each C equal to its own
    # gemm_fp4 call, tile for tile the same arithmetic.
    shapes = [(8192, 4096, 14336), (8192, 14336, 4096), (4096, 14336, 8192), (200, 296, 1056)]
    ops = [rand_operands(M, N, K, seed=11 + i) for i, (M, N, K) in enumerate(shapes)]
    sep = [m.gemm_fp4(*o, M, N, K) for o, (M, N, K) in zip(ops, shapes)]
    grouped = m.gemm_fp4_grouped([(*o, M, N, K) for o, (M, N, K) in zip(ops, shapes)])
    torch.cuda.synchronize()
    for (M, N, K), a, b in zip(shapes, sep, grouped):
        assert torch.equal(a, b), f"{M}x{N}x{K}"
    # and the ragged one against the oracle
    M, N, K = shapes[3]
    ca, sa, cb, sb = (t.cpu().numpy() for t in ops[3])
    ref = oracle.gemm_mxfp4(ca, oracle.sf_tile_to_linear(sa, M, K // 32), cb, oracle.sf_tile_to_linear(sb, N, K // 32),
                            nthreads=8)
    assert_close(grouped[3].float().cpu().numpy().astype(np.float64), ref, "grouped ragged")


def test_grouped_gemm_edge_cases(m):
    # a single descriptor; a group with an empty GEMM (skipped) and a K == 0
    # GEMM (zeros) beside a real one; results equal to gemm_fp4's
    o1 = rand_operands(384, 640, 1056, seed=5)
    c1 = m.gemm_fp4_grouped([(*o1, 384, 640, 1056)])[0]
    assert torch.equal(c1, m.gemm_fp4(*o1, 384, 640, 1056))
    o2 = rand_operands(256, 512, 512, seed=6)
    empty = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    zero_k = torch.full((128, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(1, dtype=torch.uint8, device="cuda")
    outs = m.gemm_fp4_grouped([(z, z, z, z, 0, 64, 64, empty), (*o2, 256, 512, 512), (z, z, z, z, 128, 64, 0, zero_k)])
    torch.cuda.synchronize()
    assert torch.equal(outs[1], m.gemm_fp4(*o2, 256, 512, 512))
    assert torch.count_nonzero(outs[2]).item() == 0


def test_repeated_grouped_train_step_gemms_are_bit_identical(m):
    # The grouped launch of the step's fwd, dgrad and wgrad (3 x 2.9e12 FLOP,
    # GEMMs of different K in one ring), 20 times back to back: the epilogue's
    # shared staging of a half's four warps, its named barriers and the one
    # 128-row store per block must give the same bytes every time.
    M, N, K = 8192, 4096, 14336
    specs = [(M, N, K), (M, K, N), (N, K, M)]
    ops = [rand_operands(a, b, c, seed=31 + i) for i, (a, b, c) in enumerate(specs)]
    runs = []
    for _ in range(20):
        outs = [torch.empty(a, b, dtype=torch.bfloat16, device="cuda") for a, b, _ in specs]
        m.gemm_fp4_grouped([(*o, a, b, c, out) for o, (a, b, c), out in zip(ops, specs, outs)])
        runs.append(outs)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    for i, outs in enumerate(runs[1:], 1):
        for j, (c, c0) in enumerate(zip(outs, runs[0])):
            assert torch.equal(c, c0), f"launch {i}, GEMM {j} differs from launch 0"


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_grouped_gemm_random_mixed_shapes(m, seed):
    # Four GEMMs of ragged M and N and different K per launch (a single partial
    # stage at K = 32, K tails of 32 past a 64-deep step, several stages), in
    # random order: tiles of one GEMM follow another's in the same ring, and
    # each result must equal its own gemm_fp4 call bit for bit.
    rng = np.random.default_rng(100 + seed)
    shapes = [(int(rng.integers(1, 700)), int(rng.integers(1, 700)), int(rng.choice([32, 64, 96, 160, 288, 544])))
              for _ in range(4)]
    ops = [rand_operands(M, N, K, seed=1000 * seed + i) for i, (M, N, K) in enumerate(shapes)]
    # C with a pitch rounded up to 8 elements (ragged N, aligned rows)
    out = lambda M, N: torch.empty(M, (N + 7) // 8 * 8, dtype=torch.bfloat16, device="cuda")[:, :N]
    grouped = m.gemm_fp4_grouped([(*o, M, N, K, out(M, N)) for o, (M, N, K) in zip(ops, shapes)])
    sep = [m.gemm_fp4(*o, M, N, K, c=out(M, N)) for o, (M, N, K) in zip(ops, shapes)]
    torch.cuda.synchronize()
    assert m.device_status() == 0
    for (M, N, K), a, b in zip(shapes, sep, grouped):
        assert torch.equal(a, b), f"{M}x{N}x{K}"
    # and the first one against the oracle
    M, N, K = shapes[0]
    ca, sa, cb, sb = (t.cpu().numpy() for t in ops[0])
    ref = oracle.gemm_mxfp4(ca, oracle.sf_tile_to_linear(sa, M, K // 32), cb,
                            oracle.sf_tile_to_linear(sb, N, K // 32), nthreads=8)
    assert_close(grouped[0].float().cpu().numpy().astype(np.float64), ref, f"grouped {M}x{N}x{K}")


def test_grouped_gemms_on_two_side_streams_at_once(m):
    # two grouped launches enqueued on two non-default streams, free to run
    # side by side: each result equal to its own gemm_fp4 call
    shapes_a = [(1024, 2048, 4096), (2048, 1024, 1056)]
    shapes_b = [(512, 3072, 2048), (3072, 512, 544), (256, 256, 64)]
    ops_a = [rand_operands(M, N, K, seed=70 + i) for i, (M, N, K) in enumerate(shapes_a)]
    ops_b = [rand_operands(M, N, K, seed=80 + i) for i, (M, N, K) in enumerate(shapes_b)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ga = m.gemm_fp4_grouped([(*o, M, N, K) for o, (M, N, K) in zip(ops_a, shapes_a)], stream=s1)
    gb = m.gemm_fp4_grouped([(*o, M, N, K) for o, (M, N, K) in zip(ops_b, shapes_b)], stream=s2)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    for ops, shapes, got in ((ops_a, shapes_a, ga), (ops_b, shapes_b, gb)):
        for o, (M, N, K), c in zip(ops, shapes, got):
            assert torch.equal(c, m.gemm_fp4(*o, M, N, K)), f"{M}x{N}x{K}"
