"""Pins of the MXFP8 (E4M3 + E8M0) half of the oracle against things other
than itself: hand-worked blocks (tests/golden/e4m3_blocks.txt), torch's own
float8_e4m3fn decode and round-to-nearest-even conversion (an independent
implementation of the same number format), and the format's invariants.

Method: jax-aiter README, "MXFP4 training architecture" (an FP8 dB path next
to the FP4 one); the E4M3 and scale readings are stated in the oracle source."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_pins import bf16_bits, parse_value

import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_blocks.txt")


def parse_blocks():
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
                    v, n = tok.rsplit("*", 1)
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


BLOCKS = parse_blocks()


@pytest.mark.parametrize("blk", BLOCKS, ids=[b["name"] for b in BLOCKS])
def test_golden_e4m3_block(blk):
    assert len(blk["x"]) == 32 and len(blk["codes"]) == 32 and blk["cite"]
    x = bf16_bits(blk["x"]).reshape(1, 32)
    codes, scales = oracle.cast_rows_mxfp8(x, hadamard=blk["hadamard"])
    assert scales[0, 0] == blk["scale"], f"scale {scales[0, 0]:#x} != {blk['scale']:#x}"
    assert codes[0].tolist() == blk["codes"]
    c2, s2 = oracle.cast_cols_mxfp8(np.ascontiguousarray(x.T), hadamard=blk["hadamard"])
    assert s2[0, 0] == blk["scale"] and c2[0].tolist() == blk["codes"]


def test_e4m3_values_match_torch_decode():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))          # 0x7f and 0xff only
    assert np.array_equal(mine[finite], ref[finite])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_rounding_matches_torch_rne():
    # every fp32 grid point 2^-12 apart up to 448, plus all midpoints of
    # E4M3 neighbours (the ties) and points just beside them
    grid = np.arange(0, 448 * 4096 + 1, dtype=np.float64) / 4096.0
    mags = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (mags[:-1] + mags[1:]) / 2
    eps = np.maximum(mids * 2.0 ** -20, 2.0 ** -30)
    u = np.concatenate([grid[::7], mids, mids - eps, mids + eps]).astype(np.float32)
    u = u[u <= 448.0]
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(int)
    mine = np.array([oracle.e4m3_magnitude_code(float(v)) for v in u])
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at u={u[bad[0]]!r}: {mine[bad[0]]} vs {ref[bad[0]]}"


def test_saturation_and_scale_rule():
    assert oracle.e4m3_magnitude_code(448.0) == 0x7E
    assert oracle.e4m3_magnitude_code(1e30) == 0x7E
    assert oracle.block_exponent_e4m3(448.0) == 0
    assert oracle.block_exponent_e4m3(447.9) == 0
    assert oracle.block_exponent_e4m3(256.0) == 0
    assert oracle.block_exponent_e4m3(255.9) == -1
    assert oracle.block_exponent_e4m3(0.0) == -127
    assert oracle.block_exponent_e4m3(2.0 ** 200) == 127


def test_invariants_on_random_blocks():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    codes, scales = oracle.cast_rows_mxfp8(xb)
    deq = oracle.dequant_rows_mxfp8(codes, scales)
    xf = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(64):
        for b in range(8):
            blk = xf[r, 32 * b:32 * b + 32]
            e = int(scales[r, b]) - 127
            amax = np.abs(blk).max()
            assert 2.0 ** 8 <= amax / 2.0 ** e < 2.0 ** 9             # scaled amax in [256, 512)
            d = deq[r, 32 * b:32 * b + 32]
            v = blk / 2.0 ** e
            # error at most half an E4M3 step at v's binade, except saturated values
            step = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6))) - 3))
            ok = (np.abs(v) >= 448) | (np.abs(d / 2.0 ** e - v) <= step / 2)
            assert ok.all()
            assert np.all(np.abs(d / 2.0 ** e) <= 448)


def test_gemm_mxfp8_equals_dequantized_product():
    rng = np.random.default_rng(6)
    a = (rng.standard_normal((8, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (rng.standard_normal((5, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ca, sa = oracle.cast_rows_mxfp8(a)
    cb, sb = oracle.cast_rows_mxfp8(b)
    c = oracle.gemm_mxfp8(ca, sa, cb, sb)
    da, db = oracle.dequant_rows_mxfp8(ca, sa), oracle.dequant_rows_mxfp8(cb, sb)
    # brute force in exact rational arithmetic: every term is a dyadic rational
    from fractions import Fraction
    for i in range(8):
        for j in range(5):
            s = sum(Fraction(float(da[i, k])) * Fraction(float(db[j, k])) for k in range(64))
            assert float(s) == c[i, j]
