"""The tensor-core ceiling the block-scaled FP4 GEMM is measured against: an
MMA-only microbenchmark (tests/mma_ceiling.cu: back-to-back tcgen05.mma, no
loads) on this GPU.  It pins the attainable kind::mxf4 rate that the GEMM's
efficiency is quoted against: a 256 x 256 x 64 pair MMA per 128 SM cycles,
32,768 FLOP/clk/SM, four times the bf16 rate of the same benchmark, with the
NVFP4 form (mxf4nvf4, 4X scales) no faster, the time of an MMA linear in N
(N = 224, 192, 128 at the same rate), and an N = 16 MMA bounded by the
~39-cycle issue floor."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def run_benchmark(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = tmp_path / "mma_ceiling"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", str(exe),
                    os.path.join(HERE, "mma_ceiling.cu")], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=300).stdout
    res = {}
    for line in out.splitlines():
        if line.startswith("RESULT "):
            _, name, cyc, flop, err = line.split()
            res[name] = (float(cyc), float(flop), int(err))
    return res


def test_kind_mxf4_ceiling(tmp_path):
    res = run_benchmark(tmp_path)
    print("\n".join(f"{k:28s} {c:7.2f} cycles/MMA {f:8.0f} FLOP/clk/SM" for k, (c, f, _) in res.items()))
    assert all(err == 0 for _, _, err in res.values())
    for pairs in [k.rsplit("_", 1)[1] for k in res if k.startswith("mxf4_n256")]:
        mxf4 = res[f"mxf4_n256_{pairs}"][1]
        assert 0.97 * 32768 <= mxf4 <= 1.03 * 32768
        assert abs(res[f"bf16_n256_{pairs}"][1] * 4 / mxf4 - 1) < 0.03          # fp4 = 4 x bf16 here
        assert abs(res[f"mxf8f6f4_n256_{pairs}"][1] * 2 / mxf4 - 1) < 0.03      # fp8 = 2 x bf16
        assert res[f"mxf4nvf4_4x_n256_{pairs}"][1] <= 1.03 * mxf4               # NVFP4 form no faster
        for n in (224, 192, 128):                                               # time linear in N
            assert abs(res[f"mxf4_n{n}_{pairs}"][1] / mxf4 - 1) < 0.03
        assert 30 <= res[f"mxf4_n16_{pairs}"][0] <= 60                          # issue-bound floor
