"""Pins for the oracle against things other than itself: hand-worked blocks,
closed forms, an independent construction of the Hadamard matrix, exact
rational arithmetic for tiny GEMMs, and invariants of the format.

Format and method: jax-aiter README, "Supported ops" table (MXFP4 Cast:
E2M1 + E8M0 block scales with a transposed copy; FP4 GEMM low-level:
fp4x2 codes with e8m0 scales; FP4 GEMM training: FP4 fwd / dA / dB) and
"Quick start" (grad_out cast with a Hadamard transform).
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_blocks.txt")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits(values):
    """Round-trip check: every golden value must be exactly representable."""
    out = []
    for v in values:
        u = struct.unpack("<I", struct.pack("<f", v))[0]
        if not math.isnan(v):
            assert u & 0xFFFF == 0, f"{v} is not a bf16 value"
        out.append((u >> 16) if not math.isnan(v) else 0x7FC0)
    return np.array(out, dtype=np.uint16)


def parse_value(tok):
    t = tok.strip()
    if t.lower().lstrip("-+").startswith("0x"):
        return float.fromhex(t)
    return float(t)


def parse_golden():
    blocks, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = {"name": line.strip("[]")}
            blocks.append(cur)
            continue
        key, _, val = line.partition(":")
        val = val.strip()
        if key == "x":
            xs = []
            for tok in val.split():
                if "*" in tok:
                    v, n = tok.split("*")
                    xs += [parse_value(v)] * int(n)
                else:
                    xs.append(parse_value(tok))
            cur["x"] = xs
        elif key == "scale":
            cur["scale"] = int(val, 16)
        elif key == "codes":
            cur["codes"] = [int(b, 16) for b in val.split()]
        elif key == "hadamard":
            cur["hadamard"] = bool(int(val))
        else:
            cur[key] = val
    return blocks


GOLDEN_BLOCKS = parse_golden()


@pytest.mark.parametrize("blk", GOLDEN_BLOCKS, ids=[b["name"] for b in GOLDEN_BLOCKS])
def test_golden_block(blk):
    assert len(blk["x"]) == 32 and len(blk["codes"]) == 16 and blk["cite"]
    x = bf16_bits(blk["x"]).reshape(1, 32)
    codes, scales = oracle.cast_rows(x, hadamard=blk["hadamard"])
    assert scales[0, 0] == blk["scale"], f"scale {scales[0,0]:#x} != {blk['scale']:#x}"
    assert codes[0].tolist() == blk["codes"]
    # The column-wise cast of the transposed block gives the same answer.
    c2, s2 = oracle.cast_cols(np.ascontiguousarray(x.T), hadamard=blk["hadamard"])
    assert s2[0, 0] == blk["scale"] and c2[0].tolist() == blk["codes"]


def threshold_code(u):
    """E2M1 magnitude code by counting decision boundaries passed.  The
    boundary between codes i and i+1 is the midpoint of their grid values; a
    value exactly on it goes to whichever of the two codes is even."""
    bounds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    code = 0
    for i, b in enumerate(bounds):
        if u > b or (u == b and (i + 1) % 2 == 0):
            code += 1
    return code


def test_e2m1_rounding_sweep():
    us = [k / 1024.0 for k in range(0, 8 * 1024 + 1)]
    us += [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.0000001, 1e30, 5e-324]
    for u in us:
        assert oracle.e2m1_magnitude_code(u) == threshold_code(u), u


def test_e2m1_values():
    for c in range(8):
        assert oracle.e2m1_value(c) == GRID[c]
        assert oracle.e2m1_value(c | 8) == -GRID[c]


def test_block_exponent_closed_form():
    # amax in [2^p, 2^(p+1)) -> e = p - 2, clamped to [-127, 127]
    for p in range(-149, 128):
        for mant in (1.0, 1.5, 2.0 - 2.0 ** -7):
            amax = math.ldexp(mant, p)
            e = oracle.block_exponent(amax)
            assert e == max(-127, min(127, p - 2)), (p, mant)
            if p - 2 >= -127:
                assert 4.0 <= amax / 2.0 ** e < 8.0
    assert oracle.block_exponent(0.0) == -127


def sylvester_h32():
    h = np.array([[1.0]])
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    for _ in range(5):
        h = np.kron(h2, h)
    return h


def test_hadamard_matrix_and_columns():
    h = sylvester_h32()
    assert np.array_equal(h @ h.T, 32 * np.eye(32))
    c32 = np.float32(1.0 / math.sqrt(32.0))
    for i in range(32):
        e = np.zeros(32, dtype=np.float32)
        e[i] = 1.0
        y = oracle.fwht32(e)
        assert np.array_equal(y, (h[:, i].astype(np.float32) * c32).astype(np.float32))


def test_hadamard_integer_inputs_exact():
    # With small-integer inputs every butterfly sum is exact in fp32, so the
    # transform equals one fp32 rounding of (H x) * RN(1/sqrt 32).
    rng = np.random.default_rng(11)
    h = sylvester_h32()
    c32 = np.float32(1.0 / math.sqrt(32.0))
    for _ in range(200):
        x = rng.integers(-1000, 1000, size=32).astype(np.float32)
        hx = (h @ x.astype(np.float64)).astype(np.float32)  # exact integers
        assert np.array_equal(oracle.fwht32(x), hx * c32)


def test_hadamard_random_close_to_fp64_and_involutive():
    rng = np.random.default_rng(12)
    h = sylvester_h32() / math.sqrt(32.0)
    for _ in range(200):
        x = rng.standard_normal(32).astype(np.float32)
        y = oracle.fwht32(x)
        ref = h @ x.astype(np.float64)
        assert np.max(np.abs(y - ref)) <= 1e-5 * np.linalg.norm(x)
        z = oracle.fwht32(y)  # orthonormal and symmetric: applying twice is the identity
        assert np.max(np.abs(z - x)) <= 1e-5 * np.linalg.norm(x)


def random_bf16(shape, seed, outliers=True):
    import torch
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    if outliers:
        m = torch.rand(*shape, generator=g) < 0.01
        x[m] *= 50.0
    return oracle.as_bf16_bits(x.to(torch.bfloat16))


def bits_to_f64(xb):
    return (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("hadamard", [False, True])
def test_cast_invariants(hadamard):
    xb = random_bf16((64, 256), seed=5)
    codes, scales = oracle.cast_rows(xb, hadamard=hadamard)
    assert np.all(scales != 0xFF)
    deq = oracle.dequant_rows(codes, scales)
    x = bits_to_f64(xb)
    if hadamard:
        hm = sylvester_h32() / math.sqrt(32.0)
        x = (x.reshape(64, 8, 32) @ hm.T).reshape(64, 256)
    e = scales.astype(np.int64) - 127
    scale = np.repeat(2.0 ** e, 32, axis=1)
    u = deq / scale
    # every element dequantizes onto the grid times 2^e
    assert np.all(np.isin(np.abs(u), GRID))
    # the block maximum, after scaling, lies in [4, 8)
    amax = np.abs(x).reshape(64, 8, 32).max(axis=2)
    ratio = amax / 2.0 ** e
    assert np.all((ratio >= 4.0 - 1e-6) & (ratio < 8.0))
    # error is at most half a grid step, except where |v| >= 6 saturated
    v = x / scale
    half_step = np.where(np.abs(v) < 2, 0.25, np.where(np.abs(v) < 4, 0.5, 1.0))
    ok = (np.abs(v - u) <= half_step + 1e-6) | ((np.abs(v) >= 6) & (np.abs(u) == 6))
    assert np.all(ok)
    # the sign is kept
    nib = np.stack([codes & 0xF, codes >> 4], axis=2).reshape(64, 256)
    assert np.all(((nib & 8) != 0) == np.signbit(x))


def test_cast_cols_is_cast_rows_of_transpose():
    xb = random_bf16((96, 64), seed=6)
    for had in (False, True):
        c1, s1 = oracle.cast_cols(xb, hadamard=had)
        c2, s2 = oracle.cast_rows(np.ascontiguousarray(xb.T), hadamard=had)
        assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_dequant_hand_values():
    codes = np.array([[0x07 | (0xF << 4)] + [0] * 15], dtype=np.uint8)
    d = oracle.dequant_rows(codes, np.array([[0x7F]], dtype=np.uint8))
    assert d[0, 0] == 6.0 and d[0, 1] == -6.0 and np.all(d[0, 2:] == 0)
    d = oracle.dequant_rows(codes, np.array([[0x80]], dtype=np.uint8))
    assert d[0, 0] == 12.0 and d[0, 1] == -12.0
    d = oracle.dequant_rows(codes, np.array([[0x00]], dtype=np.uint8))
    assert d[0, 0] == 6.0 * 2.0 ** -127
    d = oracle.dequant_rows(codes, np.array([[0xFF]], dtype=np.uint8))
    assert np.all(np.isnan(d))


def exact_value(code, sbyte):
    mag = Fraction(GRID[code & 7])
    return (-mag if code & 8 else mag) * (Fraction(2) ** (sbyte - 127))


@pytest.mark.parametrize("m,n,k", [(3, 5, 64), (7, 2, 96), (1, 1, 32)])
def test_gemm_exact_rationals(m, n, k):
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    ca = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(0x78, 0x87, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(0x78, 0x87, size=(n, k // 32), dtype=np.uint8)
    c = oracle.gemm_mxfp4(ca, sa, cb, sb)
    assert c.shape == (m, n)

    def elem(codes, scales, r, j):
        byte = int(codes[r, j // 2])
        return exact_value(byte & 0xF if j % 2 == 0 else byte >> 4, int(scales[r, j // 32]))

    for i in range(m):
        for j in range(n):
            ref = sum(elem(ca, sa, i, t) * elem(cb, sb, j, t) for t in range(k))
            assert Fraction(c[i, j]) == ref, (i, j)


def test_gemm_permutation():
    # A = rows of a permutation of the identity (code 2 = 1.0, scale 2^0)
    k = 64
    perm = np.random.default_rng(3).permutation(k)
    ca = np.zeros((k, k // 2), dtype=np.uint8)
    for i, p in enumerate(perm):
        ca[i, p // 2] |= (2 << 4) if p % 2 else 2
    sa = np.full((k, k // 32), 0x7F, dtype=np.uint8)
    rng = np.random.default_rng(4)
    cb = rng.integers(0, 256, size=(10, k // 2), dtype=np.uint8)
    sb = rng.integers(0x70, 0x90, size=(10, k // 32), dtype=np.uint8)
    c = oracle.gemm_mxfp4(ca, sa, cb, sb)
    b = oracle.dequant_rows(cb, sb)
    assert np.array_equal(c, b[:, perm].T)


def test_gemm_threads_identical():
    rng = np.random.default_rng(8)
    a = rng.standard_normal((37, 64))
    b = rng.standard_normal((19, 64))
    assert np.array_equal(oracle.gemm_abt(a, b, 1), oracle.gemm_abt(a, b, 4))
    assert np.allclose(oracle.gemm_abt(a, b, 1), a @ b.T, rtol=1e-12, atol=1e-12)


def test_wgrad_hadamard_cancels_only_when_on_both_operands():
    # dW = dY^T X.  The transform H (orthonormal, per 32 tokens) on the token
    # dimension of both operands cancels: (H dY)^T (H X) = dY^T X.  On one
    # operand only it would not.
    import torch
    g = torch.Generator().manual_seed(9)
    M, N, K = 256, 64, 96
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    dy = torch.randn(M, N, generator=g).to(torch.bfloat16)
    xb, dyb = oracle.as_bf16_bits(x), oracle.as_bf16_bits(dy)
    exact = bits_to_f64(dyb).T @ bits_to_f64(xb)
    ca, sa = oracle.cast_cols(dyb, hadamard=True)
    cb, sb = oracle.cast_cols(xb, hadamard=True)
    both = oracle.gemm_mxfp4(ca, sa, cb, sb)
    cb0, sb0 = oracle.cast_cols(xb, hadamard=False)
    one = oracle.gemm_mxfp4(ca, sa, cb0, sb0)
    rel = lambda c: np.linalg.norm(c - exact) / np.linalg.norm(exact)
    assert rel(both) < 0.2
    assert rel(one) > 0.8


def test_sf_tile_offsets_hand_values():
    assert oracle.sf_tile_offset(0, 0, 4) == 0
    assert oracle.sf_tile_offset(1, 0, 4) == 16
    assert oracle.sf_tile_offset(32, 0, 4) == 4
    assert oracle.sf_tile_offset(0, 1, 4) == 1
    assert oracle.sf_tile_offset(127, 3, 4) == 31 * 16 + 3 * 4 + 3
    assert oracle.sf_tile_offset(0, 4, 8) == 512
    assert oracle.sf_tile_offset(128, 0, 8) == 1024
    assert oracle.sf_tile_offset(128, 0, 5) == 1024  # 5 blocks still take 2 K-tiles


def test_sf_tile_layout_is_a_bijection():
    rows, kb = 256, 8
    r, k = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    off = oracle.sf_tile_offset(r, k, kb).ravel()
    assert sorted(off.tolist()) == list(range(rows * kb))
    lin = np.random.default_rng(1).integers(0, 255, size=(200, 7), dtype=np.uint8)
    assert np.array_equal(oracle.sf_tile_to_linear(oracle.sf_linear_to_tile(lin), 200, 7), lin)
