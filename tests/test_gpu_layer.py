"""GPU parity of the layer-level MXFP4 train step (MXFP4Linear: forward,
dgrad and wgrad through the library's casts and GEMMs) against the fp64
oracle, and the weight workspace's reuse of quantized weights.

Method: jax-aiter README, "Supported ops" rows "FP4 GEMM (training)" (FP4
forward, dA and dB with BF16 in/out) and "MXFP4 Quantizer / Workspace"
(weight / activation / grad presets, quantized-weight cache by name);
"Quick start" (grad_out cast with a Hadamard transform).  The Hadamard is on
the column copies of both wgrad operands."""
import numpy as np
import pytest
import torch

import oracle
from quantization_mxfp4_cast_gb300 import synth
from tests.util import bf16_bits, build_library, gemm_tolerance_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    build_library()
    from quantization_mxfp4_cast_gb300 import layer
    return layer


def oracle_step(x, w, dy):
    """fp64 oracle of Y = X W^T, dX = dY W, dW = dY^T X through MXFP4 casts."""
    cx, sx = oracle.cast_rows(bf16_bits(x))
    cw, sw = oracle.cast_rows(bf16_bits(w))
    y = oracle.gemm_mxfp4(cx, sx, cw, sw, nthreads=8)
    cd, sd = oracle.cast_rows(bf16_bits(dy))
    cwc, swc = oracle.cast_cols(bf16_bits(w))
    dx = oracle.gemm_mxfp4(cd, sd, cwc, swc, nthreads=8)
    cdc, sdc = oracle.cast_cols(bf16_bits(dy), hadamard=True)
    cxc, sxc = oracle.cast_cols(bf16_bits(x), hadamard=True)
    dw = oracle.gemm_mxfp4(cdc, sdc, cxc, sxc, nthreads=8)
    return y, dx, dw


def close(gpu, ref, what):
    ok, excess = gemm_tolerance_ok(gpu.float().cpu().numpy(), ref)
    assert ok, f"{what}: worst excess over tolerance {excess:.3e}"


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (160, 96, 320)])
def test_linear_train_step_matches_oracle(L, M, N, K):
    x, w, dy = synth.linear_layer(M, N, K, 1.0)
    layer = L.MXFP4Linear(w.cuda(), cache_name="t")
    xd = x.cuda().requires_grad_(True)
    y = layer(xd)
    y.backward(dy.cuda())
    torch.cuda.synchronize()
    ry, rdx, rdw = oracle_step(x, w, dy)
    close(y.detach(), ry, "fwd")
    close(xd.grad, rdx, "dgrad")
    close(layer.weight.grad, rdw, "wgrad")


def test_leading_dims_are_tokens(L):
    M, N, K = 256, 128, 256
    x, w, dy = synth.linear_layer(M, N, K, 1.0)
    layer = L.MXFP4Linear(w.cuda())
    x3 = x.cuda().reshape(2, M // 2, K).requires_grad_(True)
    y3 = layer(x3)
    assert y3.shape == (2, M // 2, N)
    y3.backward(dy.cuda().reshape(2, M // 2, N))
    torch.cuda.synchronize()
    ry, rdx, rdw = oracle_step(x, w, dy)
    close(y3.detach().reshape(M, N), ry, "fwd")
    close(x3.grad.reshape(M, K), rdx, "dgrad")
    close(layer.weight.grad, rdw, "wgrad")


def test_workspace_reuses_until_the_weight_changes(L):
    M, N, K = 128, 256, 256
    x, w, _ = synth.linear_layer(M, N, K, 1.0)
    layer = L.MXFP4Linear(w.cuda(), cache_name="w0")
    xd = x.cuda()
    with torch.no_grad():
        y0 = layer(xd)
        y1 = layer(xd)                                  # same weight: cached casts
        assert layer.workspace.casts == 1
        assert torch.equal(y0, y1)
        layer.weight.mul_(-1.0)                         # in-place update bumps the version
        y2 = layer(xd)
    torch.cuda.synchronize()
    assert layer.workspace.casts == 2
    assert torch.equal(y2, -y0)                          # the sign flips exactly in MXFP4 too
    cx, sx = oracle.cast_rows(bf16_bits(x))
    cw, sw = oracle.cast_rows(bf16_bits(-w))
    close(y2, oracle.gemm_mxfp4(cx, sx, cw, sw, nthreads=8), "fwd after update")


def test_quantizer_presets_match_the_dual_cast(L):
    t = synth.normal_bf16((256, 128), 1.0, seed=9)
    for q, had in ((L.MXFP4Quantizer.for_weight(), False), (L.MXFP4Quantizer.for_activation(), True),
                   (L.MXFP4Quantizer.for_grad(), True)):
        tq = q.quantize(t.cuda())
        torch.cuda.synchronize()
        cr, sr = oracle.cast_rows(bf16_bits(t))
        cc, sc = oracle.cast_cols(bf16_bits(t), hadamard=had)
        assert np.array_equal(tq.q_row.cpu().numpy(), cr)
        assert np.array_equal(tq.sf_row.cpu().numpy(), oracle.sf_linear_to_tile(sr))
        assert np.array_equal(tq.q_col.cpu().numpy(), cc)
        assert np.array_equal(tq.sf_col.cpu().numpy(), oracle.sf_linear_to_tile(sc))


def test_stack_matches_chain_of_layers(L):
    # Layers back to back: the stack hands each GEMM its operand already cast
    # (in the producing GEMM's epilogue), a chain of MXFP4Linear layers casts
    # the bf16 tensors in between.  The fused casts equal the separate ones
    # byte for byte, so output and every gradient must be identical.
    dims = [128, 256, 96, 160]
    M = 320
    ws = [synth.normal_bf16((dims[i + 1], dims[i]), 0.05, seed=40 + i).cuda() for i in range(3)]
    x = synth.normal_bf16((M, dims[0]), 1.0, seed=50).cuda()
    dy = synth.normal_bf16((M, dims[-1]), 1e-2, seed=51).cuda()

    stack = L.MXFP4LinearStack([w.clone() for w in ws])
    xs = x.clone().requires_grad_(True)
    ys = stack(xs)
    ys.backward(dy)

    layers = [L.MXFP4Linear(w.clone(), cache_name=f"l{i}") for i, w in enumerate(ws)]
    xc = x.clone().requires_grad_(True)
    h = xc
    for layer in layers:
        h = layer(h)
    h.backward(dy)
    torch.cuda.synchronize()

    assert torch.equal(ys, h)
    assert torch.equal(xs.grad, xc.grad)
    for i, (p, layer) in enumerate(zip(stack.weights, layers)):
        assert torch.equal(p.grad, layer.weight.grad), f"dW of layer {i}"


def test_single_layer_stack_is_the_layer(L):
    M, N, K = 256, 384, 512
    w = synth.normal_bf16((N, K), 0.02, seed=60).cuda()
    x = synth.normal_bf16((M, K), 1.0, seed=61).cuda()
    dy = synth.normal_bf16((M, N), 1e-3, seed=62).cuda()
    stack, layer = L.MXFP4LinearStack([w.clone()]), L.MXFP4Linear(w.clone())
    xs, xl = x.clone().requires_grad_(True), x.clone().requires_grad_(True)
    ys, yl = stack(xs), layer(xl)
    ys.backward(dy)
    yl.backward(dy)
    torch.cuda.synchronize()
    assert torch.equal(ys, yl) and torch.equal(xs.grad, xl.grad)
    assert torch.equal(stack.weights[0].grad, layer.weight.grad)


def test_stack_inference_matches_training_forward(L):
    dims = [64, 128, 96]
    ws = [synth.normal_bf16((dims[i + 1], dims[i]), 0.05, seed=80 + i).cuda() for i in range(2)]
    x = synth.normal_bf16((160, dims[0]), 1.0, seed=82).cuda()
    stack = L.MXFP4LinearStack(ws)
    y_train = stack(x.clone().requires_grad_(True))
    with torch.no_grad():
        y_infer = stack(x)
    torch.cuda.synchronize()
    assert torch.equal(y_train.detach(), y_infer)


def test_forward_without_backward_makes_the_row_copy_only(L):
    # Without a weight gradient the activation's column copy (read only by the
    # wgrad) is not made: the row-only cast gives the dual cast's row bytes,
    # and the layer's output is the same with and without autograd.
    M, N, K = 192, 256, 320
    w = synth.normal_bf16((N, K), 0.02, seed=90).cuda()
    x = synth.normal_bf16((M, K), 1.0, seed=91).cuda()
    q = L.MXFP4Quantizer.for_activation()
    rows, dual = q.quantize_rows(x), q.quantize(x)
    torch.cuda.synchronize()
    assert rows.q_col is None and rows.sf_col is None
    assert torch.equal(rows.q_row, dual.q_row) and torch.equal(rows.sf_row, dual.sf_row)
    layer = L.MXFP4Linear(w.clone())
    y_train = layer(x)
    with torch.no_grad():
        y_infer = layer(x)
    frozen = L.MXFP4Linear(w.clone())
    frozen.weight.requires_grad_(False)
    xg = x.clone().requires_grad_(True)
    y_frozen = frozen(xg)               # dgrad still possible: no wgrad, no column copy of x
    y_frozen.backward(torch.ones_like(y_frozen))
    torch.cuda.synchronize()
    assert torch.equal(y_train.detach(), y_infer) and torch.equal(y_infer, y_frozen.detach())
    assert xg.grad is not None and torch.isfinite(xg.grad.float()).all()
