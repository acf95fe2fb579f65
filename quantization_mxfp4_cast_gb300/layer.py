"""Layer-level MXFP4 training step on top of the C ABI.

Method: jax-aiter README, "Supported ops" table, rows "FP4 GEMM (training)"
(BF16 in/out; forward, dA and dB all in FP4) and "MXFP4 Quantizer /
Workspace" (quantizer presets for weights, activations and gradients; a
workspace that caches a quantized weight under a name), and "Quick start"
(grad_out is cast with a Hadamard transform).  Readings, as in the rest of
the library: the Hadamard is applied to the column (transposed) copies of
both wgrad operands, grad_out and the activations, along the tokens, so it
cancels in dY^T X; the weight gets no transform.

Everything here is bookkeeping: every cast and GEMM runs in the library's
CUDA kernels through the binding, on the current torch stream.

    q = MXFP4Quantizer.for_weight()
    w_q = q.quantize(w)                          # MXFP4Tensor: row + column copies
    ws = WeightWorkspace()
    w_q = ws.get_or_quantize(w, q, cache_name="mlp_down")   # recast only when w changed
    y = MXFP4Linear(w, cache_name="mlp_down")(x)             # autograd: fwd, dgrad, wgrad
    y = MXFP4LinearStack([w1, w2])(x)       # layers back to back, casts fused into the GEMMs
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import gemm_fp4, gemm_fp4_cast_out, gemm_fp4_grouped, mxfp4_cast, mxfp4_cast_dual, scales_bytes


@dataclass
class MXFP4Tensor:
    """The MXFP4 copies of a bf16 matrix T[R, C]: row-wise (codes [R, C/2],
    blocks of 32 along C) and column-wise (codes [C, R/2], blocks of 32 along
    R, i.e. T^T quantized), with their tile-layout scales.  The column copy is
    None when only the row copy was made (a forward with no backward)."""
    rows: int
    cols: int
    q_row: torch.Tensor
    sf_row: torch.Tensor
    q_col: torch.Tensor
    sf_col: torch.Tensor
    hadamard_col: bool

    @staticmethod
    def empty(rows: int, cols: int, hadamard_col: bool, device) -> "MXFP4Tensor":
        u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=device)
        return MXFP4Tensor(rows, cols, u8(rows, cols // 2), u8(scales_bytes(rows, cols)),
                           u8(cols, rows // 2), u8(scales_bytes(cols, rows)), hadamard_col)


class MXFP4Quantizer:
    """What one role's dual cast produces.  `hadamard_col`: the column copy
    (the one a wgrad contracts over the tokens) gets the 32-point transform."""

    def __init__(self, role: str, hadamard_col: bool):
        self.role = role
        self.hadamard_col = hadamard_col

    @classmethod
    def for_weight(cls) -> "MXFP4Quantizer":
        """W[N, K]: row copy for fwd (contraction over K), column copy for
        dgrad (contraction over N); no transform."""
        return cls("weight", hadamard_col=False)

    @classmethod
    def for_activation(cls) -> "MXFP4Quantizer":
        """X[M, K]: row copy for fwd, column copy (Hadamard along M) for wgrad."""
        return cls("activation", hadamard_col=True)

    @classmethod
    def for_grad(cls) -> "MXFP4Quantizer":
        """dY[M, N]: row copy for dgrad, column copy (Hadamard along M) for wgrad."""
        return cls("grad", hadamard_col=True)

    def quantize_rows(self, t: torch.Tensor) -> MXFP4Tensor:
        """Only the row copy of the 2-D bf16 t (what a forward GEMM reads):
        one row-wise cast, no transposed copy."""
        if t.dim() != 2:
            raise ValueError("quantize_rows expects a 2-D tensor")
        R, C = t.shape
        q, sf = mxfp4_cast(t, stream=torch.cuda.current_stream(t.device))
        return MXFP4Tensor(R, C, q, sf, None, None, self.hadamard_col)

    def quantize(self, t: torch.Tensor, out: MXFP4Tensor | None = None) -> MXFP4Tensor:
        """One dual cast of the 2-D bf16 t (rows and columns multiples of 32)."""
        if t.dim() != 2:
            raise ValueError("quantize expects a 2-D tensor")
        R, C = t.shape
        if out is None or (out.rows, out.cols) != (R, C):
            out = MXFP4Tensor.empty(R, C, self.hadamard_col, t.device)
        out.hadamard_col = self.hadamard_col
        mxfp4_cast_dual(t, hadamard_col=self.hadamard_col,
                        out=(out.q_row, out.sf_row, out.q_col, out.sf_col),
                        stream=torch.cuda.current_stream(t.device))
        return out


class WeightWorkspace:
    """Cache of quantized weights by name.  An entry is reused while the
    weight is the same storage at the same version (torch bumps a tensor's
    version on every in-place update, e.g. an optimizer step) with the same
    shape and quantizer role; otherwise it is recast into the entry's buffers."""

    def __init__(self):
        self._entries: dict = {}
        self.casts = 0  # number of casts done (for tests and reporting)

    def get_or_quantize(self, w: torch.Tensor, quantizer: MXFP4Quantizer,
                        cache_name: str | None = None) -> MXFP4Tensor:
        name = cache_name if cache_name is not None else f"_anon_{id(w)}"
        key = (w.data_ptr(), w._version, tuple(w.shape), quantizer.role, quantizer.hadamard_col)
        entry = self._entries.get(name)
        if entry is not None and entry[0] == key:
            return entry[1]
        out = quantizer.quantize(w, out=entry[1] if entry is not None else None)
        self.casts += 1
        self._entries[name] = (key, out)
        return out

    def invalidate(self, cache_name: str | None = None):
        """Drop one entry, or all of them."""
        if cache_name is None:
            self._entries.clear()
        else:
            self._entries.pop(cache_name, None)


class _MXFP4LinearFn(torch.autograd.Function):
    """y = x w^T with fwd, dgrad and wgrad in MXFP4 (fp32 accumulation, bf16 out)."""

    @staticmethod
    def forward(ctx, x2, w, w_q, act_q, grad_q):
        M, K = x2.shape
        N = w.shape[0]
        # the column copy of x serves only the wgrad: without a weight gradient
        # (inference, or a frozen weight) the row-wise cast alone is made
        x_q = act_q.quantize(x2) if ctx.needs_input_grad[1] else act_q.quantize_rows(x2)
        stream = torch.cuda.current_stream(x2.device)
        y = gemm_fp4(x_q.q_row, x_q.sf_row, w_q.q_row, w_q.sf_row, M, N, K, stream=stream)
        ctx.x_q, ctx.w_q, ctx.grad_q = x_q, w_q, grad_q
        ctx.shape = (M, N, K)
        return y

    @staticmethod
    def backward(ctx, dy):
        M, N, K = ctx.shape
        dy = dy.contiguous()
        dy_q = ctx.grad_q.quantize(dy)
        stream = torch.cuda.current_stream(dy.device)
        gemms = {}
        if ctx.needs_input_grad[0]:
            # dX[M,K] = dY[M,N] . W[N,K]: row(dY) against col(W), contraction over N
            gemms["dx"] = (dy_q.q_row, dy_q.sf_row, ctx.w_q.q_col, ctx.w_q.sf_col, M, K, N)
        if ctx.needs_input_grad[1]:
            # dW[N,K] = dY^T . X: col(dY) against col(X), contraction over the tokens M
            gemms["dw"] = (dy_q.q_col, dy_q.sf_col, ctx.x_q.q_col, ctx.x_q.sf_col, N, K, M)
        # both backward GEMMs in one launch
        outs = dict(zip(gemms, gemm_fp4_grouped(gemms.values(), stream=stream))) if gemms else {}
        return outs.get("dx"), outs.get("dw"), None, None, None


def mxfp4_linear(x: torch.Tensor, w: torch.Tensor, w_q: MXFP4Tensor | None = None,
                 workspace: WeightWorkspace | None = None, cache_name: str | None = None) -> torch.Tensor:
    """y = x w^T for bf16 x[..., K] and w[N, K] with MXFP4 fwd, dgrad and
    wgrad.  The tokens (x's leading dimensions, flattened) and N, K must be
    multiples of 32.  The weight's casts come from `w_q`, else from
    `workspace` (cached under `cache_name`), else are made here."""
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise ValueError("mxfp4_linear expects bf16 tensors")
    x2 = x.reshape(-1, x.shape[-1])
    if not x2.is_contiguous():
        x2 = x2.contiguous()
    if w_q is None:
        wq = MXFP4Quantizer.for_weight()
        w_q = workspace.get_or_quantize(w, wq, cache_name) if workspace is not None else wq.quantize(w)
    y = _MXFP4LinearFn.apply(x2, w, w_q, MXFP4Quantizer.for_activation(), MXFP4Quantizer.for_grad())
    return y.reshape(*x.shape[:-1], w.shape[0])


class MXFP4Linear(torch.nn.Module):
    """A bias-free linear layer whose training step runs in MXFP4.  The weight's
    quantized copies are cached in `workspace` and recast only after the weight
    changes (e.g. once per optimizer step, not once per micro-batch)."""

    def __init__(self, weight: torch.Tensor, cache_name: str = "linear",
                 workspace: WeightWorkspace | None = None):
        super().__init__()
        self.weight = torch.nn.Parameter(weight)
        self.cache_name = cache_name
        self.workspace = workspace if workspace is not None else WeightWorkspace()

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return mxfp4_linear(x, self.weight, workspace=self.workspace, cache_name=self.cache_name)


class _MXFP4StackFn(torch.autograd.Function):
    """y = x W_0^T W_1^T ... W_{L-1}^T, layers back to back with nothing in
    between, every GEMM in MXFP4.  Each forward GEMM but the last writes, in
    its epilogue, the next layer's activation casts instead of a bf16 output;
    each dgrad but the first writes the casts of dX that the layer below takes
    as its grad_out.  So the only separate casts are those of the input and of
    the incoming gradient, and the numbers are those of a chain of
    MXFP4Linear layers: a fused cast equals the separate cast of the bf16
    tensor it replaces, byte for byte.  The saved activations are their
    quantized copies (what wgrad reads), not bf16 tensors."""

    @staticmethod
    def forward(ctx, x2, w_qs, *ws):
        M = x2.shape[0]
        stream = torch.cuda.current_stream(x2.device)
        # without a backward only the row copies are made (the column copies
        # serve the wgrads)
        train = any(ctx.needs_input_grad)
        act = MXFP4Quantizer.for_activation()
        x_q = act.quantize(x2) if train else act.quantize_rows(x2)
        acts, y = [], None
        for i, (w, w_q) in enumerate(zip(ws, w_qs)):
            N, K = w.shape
            acts.append(x_q)
            if i + 1 < len(ws):
                nxt = MXFP4Tensor.empty(M, N, True, x2.device)
                if not train:
                    nxt.q_col = nxt.sf_col = None
                gemm_fp4_cast_out(x_q.q_row, x_q.sf_row, w_q.q_row, w_q.sf_row, M, N, K, hadamard_col=True,
                                  out=(nxt.q_row, nxt.sf_row, nxt.q_col, nxt.sf_col), write_c=False,
                                  stream=stream)
                x_q = nxt
            else:
                y = gemm_fp4(x_q.q_row, x_q.sf_row, w_q.q_row, w_q.sf_row, M, N, K, stream=stream)
        if any(ctx.needs_input_grad):  # keep the quantized activations only for a backward
            ctx.acts, ctx.w_qs, ctx.shapes, ctx.M = acts, w_qs, [tuple(w.shape) for w in ws], M
        return y

    @staticmethod
    def backward(ctx, dy):
        M, L = ctx.M, len(ctx.w_qs)
        stream = torch.cuda.current_stream(dy.device)
        dy_q = MXFP4Quantizer.for_grad().quantize(dy.contiguous())
        dws, dx = [None] * L, None
        for i in reversed(range(L)):
            N, K = ctx.shapes[i]
            x_q, w_q = ctx.acts[i], ctx.w_qs[i]
            if i == 0:
                # the first layer: its wgrad and dgrad (bf16 dX) in one launch
                gemms = {}
                if ctx.needs_input_grad[2]:
                    gemms["dw"] = (dy_q.q_col, dy_q.sf_col, x_q.q_col, x_q.sf_col, N, K, M)
                if ctx.needs_input_grad[0]:
                    gemms["dx"] = (dy_q.q_row, dy_q.sf_row, w_q.q_col, w_q.sf_col, M, K, N)
                outs = dict(zip(gemms, gemm_fp4_grouped(gemms.values(), stream=stream))) if gemms else {}
                dws[0], dx = outs.get("dw"), outs.get("dx")
                break
            if ctx.needs_input_grad[2 + i]:
                # dW_i[N,K] = dY_i^T . X_i, contraction over the tokens
                dws[i] = gemm_fp4(dy_q.q_col, dy_q.sf_col, x_q.q_col, x_q.sf_col, N, K, M, stream=stream)
            # dX_i = dY_i . W_i is the grad_out of layer i-1: only its casts
            nxt = MXFP4Tensor.empty(M, K, True, dy.device)
            gemm_fp4_cast_out(dy_q.q_row, dy_q.sf_row, w_q.q_col, w_q.sf_col, M, K, N, hadamard_col=True,
                              out=(nxt.q_row, nxt.sf_row, nxt.q_col, nxt.sf_col), write_c=False,
                              stream=stream)
            dy_q = nxt
        return (dx, None, *dws)


class MXFP4LinearStack(torch.nn.Module):
    """Bias-free linear layers applied back to back (weights W_i[N_i, K_i] with
    K_{i+1} = N_i, nothing between them) whose training step runs in MXFP4,
    each GEMM handing the next one its operand already quantized.  The
    weights' casts are cached in `workspace` like MXFP4Linear's.  Every
    dimension, and the number of tokens, must be a multiple of 32."""

    def __init__(self, weights, cache_prefix: str = "stack", workspace: WeightWorkspace | None = None):
        super().__init__()
        if len(weights) == 0:
            raise ValueError("MXFP4LinearStack needs at least one weight")
        for i, w in enumerate(weights):
            if w.dim() != 2 or w.shape[0] % 32 or w.shape[1] % 32:
                raise ValueError(f"weight {i}: expected [N, K] with N, K multiples of 32, got {tuple(w.shape)}")
            if i and w.shape[1] != weights[i - 1].shape[0]:
                raise ValueError(f"weight {i} takes {w.shape[1]} inputs, weight {i - 1} gives {weights[i - 1].shape[0]}")
        self.weights = torch.nn.ParameterList([torch.nn.Parameter(w) for w in weights])
        self.cache_prefix = cache_prefix
        self.workspace = workspace if workspace is not None else WeightWorkspace()

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise ValueError("MXFP4LinearStack expects bf16 input")
        x2 = x.reshape(-1, x.shape[-1])
        if not x2.is_contiguous():
            x2 = x2.contiguous()
        if x2.shape[0] % 32:
            raise ValueError("the number of tokens must be a multiple of 32")
        wq = MXFP4Quantizer.for_weight()
        w_qs = [self.workspace.get_or_quantize(w, wq, f"{self.cache_prefix}.{i}") for i, w in enumerate(self.weights)]
        y = _MXFP4StackFn.apply(x2, w_qs, *self.weights)
        return y.reshape(*x.shape[:-1], y.shape[-1])
