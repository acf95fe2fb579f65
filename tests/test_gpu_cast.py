"""GPU parity of the MXFP4 cast kernels against the oracle: codes and scales
must match bit for bit (jax-aiter README, "Supported ops", MXFP4 Cast row:
CastMxfp4JA row-wise, CastMxfp4DualJA row + transposed; "Quick start": grad
cast with a Hadamard transform)."""
import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.test_oracle_pins import GOLDEN_BLOCKS, bf16_bits as golden_bits
from tests.util import bf16_bits, build_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    build_library()
    import quantization_mxfp4_cast_gb300 as mod
    return mod


def tile_to_lin(sf_gpu, rows, cols):
    return oracle.sf_tile_to_linear(sf_gpu.cpu().numpy(), rows, cols // 32)


def check_row(m, x, hadamard, linear):
    q, sf = m.mxfp4_cast(x.cuda(), hadamard=hadamard, linear_scales=linear)
    torch.cuda.synchronize()
    codes, scales = oracle.cast_rows(bf16_bits(x), hadamard=hadamard)
    R, C = x.shape
    got_sf = sf.cpu().numpy().reshape(R, C // 32) if linear else tile_to_lin(sf, R, C)
    assert np.array_equal(got_sf, scales), "scales differ"
    assert np.array_equal(q.cpu().numpy(), codes), "codes differ"
    if not linear:  # padding bytes of the tiled layout are written as zero
        full = oracle.sf_linear_to_tile(scales)
        assert np.array_equal(sf.cpu().numpy(), full)


def check_dual(m, x, had_row, had_col, linear):
    qr, sr, qc, sc = m.mxfp4_cast_dual(x.cuda(), hadamard_row=had_row, hadamard_col=had_col,
                                       linear_scales=linear)
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    R, C = x.shape
    cr, srr = oracle.cast_rows(xb, hadamard=had_row)
    cc, scc = oracle.cast_cols(xb, hadamard=had_col)
    if linear:
        assert np.array_equal(sr.cpu().numpy().reshape(R, C // 32), srr)
        assert np.array_equal(sc.cpu().numpy().reshape(C, R // 32), scc)
    else:
        assert np.array_equal(sr.cpu().numpy(), oracle.sf_linear_to_tile(srr))
        assert np.array_equal(sc.cpu().numpy(), oracle.sf_linear_to_tile(scc))
    assert np.array_equal(qr.cpu().numpy(), cr)
    assert np.array_equal(qc.cpu().numpy(), cc)


SHAPES = [(256, 512), (128, 128), (96, 160), (1, 32), (300, 224), (640, 384)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("linear", [False, True])
def test_row_cast_parity(m, shape, hadamard, linear):
    x = synth.with_outliers(synth.normal_bf16(shape, 1.0, seed=shape[0] + shape[1]), frac=0.01)
    check_row(m, x, hadamard, linear)


DUAL_SHAPES = [(256, 512), (128, 128), (96, 160), (32, 32), (320, 224), (640, 384)]


@pytest.mark.parametrize("shape", DUAL_SHAPES)
@pytest.mark.parametrize("had", [(False, False), (True, True), (False, True)])
@pytest.mark.parametrize("linear", [False, True])
def test_dual_cast_parity(m, shape, had, linear):
    x = synth.with_outliers(synth.normal_bf16(shape, 1.0, seed=7 * shape[0] + shape[1]), frac=0.01)
    check_dual(m, x, had[0], had[1], linear)


def test_golden_blocks_on_gpu(m):
    for blk in GOLDEN_BLOCKS:
        bits = golden_bits(blk["x"]).reshape(1, 32)
        x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        q, sf = m.mxfp4_cast(x.cuda(), hadamard=blk["hadamard"], linear_scales=True)
        torch.cuda.synchronize()
        assert sf.cpu().numpy()[0] == blk["scale"], blk["name"]
        assert q.cpu().numpy()[0].tolist() == blk["codes"], blk["name"]
        # the same block as a column (32 rows x 1 column, padded to 32 columns)
        xc = torch.zeros(32, 32, dtype=torch.bfloat16)
        xc[:, 0] = x[0]
        _, _, qc, sc = m.mxfp4_cast_dual(xc.cuda(), hadamard_col=blk["hadamard"], linear_scales=True)
        torch.cuda.synchronize()
        assert sc.cpu().numpy()[0] == blk["scale"], blk["name"]
        assert qc.cpu().numpy()[0].tolist() == blk["codes"], blk["name"]


@pytest.mark.parametrize("hadamard", [False, True])
def test_exhaustive_bf16_patterns(m, hadamard):
    # every one of the 65536 bf16 bit patterns, in natural order and in four
    # seeded permutations, as blocks of 32 -- both directions
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    arrs = [pats] + [np.random.default_rng(s).permutation(pats) for s in range(4)]
    bits = np.concatenate(arrs).reshape(-1, 256)  # 1280 x 256
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    check_dual(m, x, hadamard, hadamard, linear=False)


def test_full_size_cast_config(m):
    # activations [8192, 4096] ~ N(0,1) with 0.1% x50 outliers, dual, Hadamard off and on
    x = synth.cast_input()
    for had in (False, True):
        check_dual(m, x, had, had, linear=False)


def test_side_stream_ordering(m):
    # work queued ahead on a side stream must finish before the cast reads x
    s = torch.cuda.Stream()
    ballast = torch.randn(4096, 4096, device="cuda")
    x_host = synth.normal_bf16((2048, 1024), 1.0, seed=21)
    x = torch.zeros(2048, 1024, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        for _ in range(8):
            ballast = ballast @ ballast * 1e-3
        x.copy_(x_host.cuda(non_blocking=False))
        q, sf = m.mxfp4_cast(x, stream=s)
    s.synchronize()
    codes, scales = oracle.cast_rows(bf16_bits(x_host))
    assert np.array_equal(q.cpu().numpy(), codes)
    assert np.array_equal(tile_to_lin(sf, 2048, 1024), scales)


def test_pitched_input(m):
    big = synth.normal_bf16((192, 320), 1.0, seed=33).cuda()
    view = big[:, 32:288]  # ldx = 320, 16-byte aligned start
    q, sf = m.mxfp4_cast(view)
    torch.cuda.synchronize()
    codes, scales = oracle.cast_rows(bf16_bits(view.contiguous()))
    assert np.array_equal(q.cpu().numpy(), codes)
    assert np.array_equal(tile_to_lin(sf, 192, 256), scales)


@pytest.mark.parametrize("shape", [(2432, 4096), (1280, 2048), (4096, 512)])
def test_whole_rounds_and_short_tails(m, shape):
    # 608 tiles = 4 whole rounds of 152 CTAs (no tail); 160 tiles = one round
    # and 8 tiles dealt out slab by slab; 128 tiles: every slab a tail slab
    x = synth.with_outliers(synth.normal_bf16(shape, 1.0, seed=shape[0] + shape[1]), frac=0.01)
    check_dual(m, x, False, True, linear=False)
    check_row(m, x, False, linear=False)


def test_same_stream_ordering(m):
    # Casts are launched with programmatic stream serialization: a cast may
    # begin while the previous kernel in the stream finishes, but must not read
    # its input or write its outputs before that kernel is done.  (1) a torch
    # kernel writes x, the cast reads it right after; (2) two casts write the
    # same outputs back to back: the second's bytes must win everywhere.
    R, C = 1024, 2048
    a = synth.normal_bf16((R, C), 1.0, seed=41)
    b = synth.normal_bf16((R, C), 1e-3, seed=42)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        src = a.cuda()
        x = torch.empty_like(src)
        for _ in range(3):
            torch.mul(src, 1.0, out=x)  # the input is produced by the kernel just before the cast
        out = m.mxfp4_cast_dual(x, hadamard_col=True, stream=s)
        xb = b.cuda()
        for _ in range(4):
            m.mxfp4_cast_dual(x, hadamard_col=True, out=out, stream=s)
            m.mxfp4_cast_dual(xb, hadamard_col=True, out=out, stream=s)
    s.synchronize()
    cr, srr = oracle.cast_rows(bf16_bits(b))
    cc, scc = oracle.cast_cols(bf16_bits(b), hadamard=True)
    assert np.array_equal(out[0].cpu().numpy(), cr) and np.array_equal(out[2].cpu().numpy(), cc)
    assert np.array_equal(out[1].cpu().numpy(), oracle.sf_linear_to_tile(srr))
    assert np.array_equal(out[3].cpu().numpy(), oracle.sf_linear_to_tile(scc))
    q, _ = m.mxfp4_cast(x, stream=s)
    s.synchronize()
    assert np.array_equal(q.cpu().numpy(), oracle.cast_rows(bf16_bits(a))[0])


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_and_flags(m, seed):
    # Seeded random shapes (rows and columns multiples of 32, from one slab to
    # a few dozen tiles, so the grid's whole rounds, the slab-by-slab tail and
    # the tile-staged and direct scale paths all occur), random Hadamard flags
    # and scale layout, activations with outliers: every code and scale byte
    # equal to the oracle's.
    rng = np.random.default_rng(500 + seed)
    R = 32 * int(rng.integers(1, 80))
    C = 32 * int(rng.integers(1, 80))
    had_row, had_col, linear = (bool(v) for v in rng.integers(0, 2, size=3))
    x = synth.with_outliers(synth.normal_bf16((R, C), float(rng.choice([1e-3, 0.02, 1.0])), seed=600 + seed),
                            frac=0.001)
    check_dual(m, x, had_row, had_col, linear)
    check_row(m, x, had_row, linear)


def filled_dual_outputs(x, fill=0xAB):
    # outputs pre-filled with a byte the cast never leaves behind, so every
    # byte the two paths write (and every byte they leave alone) is compared
    R, C = x.shape
    import quantization_mxfp4_cast_gb300 as mod
    u8 = lambda *s: torch.full(s, fill, dtype=torch.uint8, device=x.device)
    return (u8(R, C // 2), u8(mod.scales_bytes(R, C)), u8(C, R // 2), u8(mod.scales_bytes(C, R)))


def check_grouped_against_separate(m, items):
    """items: (x, had_row, had_col) on the GPU.  The grouped call's bytes must
    equal those of one mxfp4_cast_dual call per item."""
    got = m.mxfp4_cast_dual_grouped([(x, hr, hc, filled_dual_outputs(x)) for x, hr, hc in items])
    for (x, hr, hc), g in zip(items, got):
        ref = m.mxfp4_cast_dual(x, hadamard_row=hr, hadamard_col=hc, out=filled_dual_outputs(x))
        torch.cuda.synchronize()
        for a, b, name in zip(g, ref, ("q_row", "sf_row", "q_col", "sf_col")):
            assert torch.equal(a, b), f"{tuple(x.shape)} had_row={hr} had_col={hc}: {name} differs"
    return got


def test_grouped_dual_cast_step_shapes(m):
    # the train step's three casts (X and dY with the column Hadamard, W
    # without) in one launch, at a quarter of the token count
    x = synth.normal_bf16((2048, 14336), 0.02, seed=1).cuda()
    w = synth.normal_bf16((4096, 14336), 0.02, seed=2).cuda()
    dy = synth.normal_bf16((2048, 4096), 1e-3, seed=3).cuda()
    check_grouped_against_separate(m, [(x, False, True), (w, False, False), (dy, False, True)])


def test_grouped_dual_cast_against_oracle(m):
    # mixed shapes (ragged tiles, one slab, four casts) and every flag pair,
    # checked byte for byte against the oracle
    items = [(synth.with_outliers(synth.normal_bf16(s, 1.0, seed=70 + k), frac=0.01), hr, hc)
             for k, (s, hr, hc) in enumerate([((96, 160), False, True), ((32, 32), True, True),
                                              ((320, 224), False, False), ((256, 512), True, False)])]
    got = m.mxfp4_cast_dual_grouped([(x.cuda(), hr, hc) for x, hr, hc in items])
    torch.cuda.synchronize()
    for (x, hr, hc), (qr, sr, qc, sc) in zip(items, got):
        xb = bf16_bits(x)
        cr, srr = oracle.cast_rows(xb, hadamard=hr)
        cc, scc = oracle.cast_cols(xb, hadamard=hc)
        assert np.array_equal(qr.cpu().numpy(), cr)
        assert np.array_equal(qc.cpu().numpy(), cc)
        assert np.array_equal(sr.cpu().numpy(), oracle.sf_linear_to_tile(srr))
        assert np.array_equal(sc.cpu().numpy(), oracle.sf_linear_to_tile(scc))


@pytest.mark.parametrize("seed", range(4))
def test_grouped_dual_cast_random(m, seed):
    # 1-4 casts of random shapes (multiples of 32, up to a few dozen tiles)
    # and random Hadamard flags, with an empty cast among them now and then
    rng = np.random.default_rng(900 + seed)
    n = int(rng.integers(1, 5))
    items = []
    for k in range(n):
        R, C = 32 * int(rng.integers(1, 70)), 32 * int(rng.integers(1, 70))
        if rng.random() < 0.15:
            R = 0
        x = synth.with_outliers(synth.normal_bf16((max(R, 32), C), float(rng.choice([1e-3, 1.0])),
                                                  seed=950 + 10 * seed + k), frac=0.001)[:R].cuda()
        items.append((x, bool(rng.integers(0, 2)), bool(rng.integers(0, 2))))
    nonempty = [it for it in items if it[0].shape[0] > 0]
    if nonempty:
        check_grouped_against_separate(m, nonempty)
    m.mxfp4_cast_dual_grouped([(x, hr, hc) for x, hr, hc in items])  # empty ones are skipped
    torch.cuda.synchronize()


def test_grouped_dual_cast_repeated_bit_identical(m):
    # thirty back-to-back grouped launches of the step's three casts (full
    # size: every SM runs many tiles, so the column-code staging buffers
    # and the scale-tile buffers are reused many times over): every byte of
    # every launch equal to the first launch's
    x = synth.normal_bf16((8192, 14336), 0.02, seed=11).cuda()
    w = synth.normal_bf16((4096, 14336), 0.02, seed=12).cuda()
    dy = synth.normal_bf16((8192, 4096), 1e-3, seed=13).cuda()
    items = [(x, False, True), (w, False, False), (dy, False, True)]
    first = [tuple(t.clone() for t in o) for o in m.mxfp4_cast_dual_grouped(items)]
    outs = [filled_dual_outputs(t) for t, _, _ in items]
    for rep in range(30):
        m.mxfp4_cast_dual_grouped([(t, hr, hc, o) for (t, hr, hc), o in zip(items, outs)])
        torch.cuda.synchronize()
        for k, (o, f) in enumerate(zip(outs, first)):
            for a, b in zip(o, f):
                assert torch.equal(a, b), f"launch {rep}, cast {k} differs"
    assert m.device_status() == 0
