"""Shared test helpers: bit views, the GEMM tolerance, library build."""
import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float64)


def gemm_tolerance_ok(gpu: np.ndarray, ref: np.ndarray, rms_ref: float = None):
    """|gpu - oracle| <= 2^-8 |oracle| + 1e-3 rms(oracle), elementwise; rms over
    all the oracle values given unless supplied.  Returns (ok, worst excess)."""
    ref = np.asarray(ref, dtype=np.float64)
    gpu = np.asarray(gpu, dtype=np.float64)
    if rms_ref is None:
        rms_ref = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms_ref
    err = np.abs(gpu - ref)
    finite = np.isfinite(gpu).all()
    excess = float(np.max(err - bound)) if ref.size else 0.0
    return bool(finite and np.all(err <= bound)), excess


def build_library():
    from quantization_mxfp4_cast_gb300 import build
    return build.build()
