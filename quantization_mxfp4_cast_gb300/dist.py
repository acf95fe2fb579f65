"""Data-parallel (FSDP-style) wgrad: token-sharded MXFP4 dW partials summed by
a reduce-scatter.

Method: jax-aiter README, "Supported ops" row "FP4 GEMM (training)" (FP4 dB
with FSDP-aware wgrad sharding), "Quick start" (FP4 dB: NT wgrad with
FSDP-aware psum sharding) and "MXFP4 training architecture" (dB overlapped
with the FSDP communication).

Each rank holds a contiguous shard of the tokens, X_r[M_r, K] and dY_r[M_r, N].
Its wgrad GEMM dW_r = dY_r^T . X_r contracts over its own tokens only; the
weight gradient is the sum over ranks.  Under FSDP each weight is kept
row-sharded, so the sum is a reduce-scatter: rank r receives rows
[r N / P, (r + 1) N / P) of sum_r dW_r.

Readings, where the pages are silent:
  * shard boundaries fall on multiples of 32 tokens, so no 32-element block
    of the column casts (the wgrad operands, quantized along the tokens, with
    the 32-point Hadamard) straddles two ranks: the shards' casts are exactly
    the full tensor's casts, split, and sum_r dW_r is the unsharded wgrad of
    the dequantized operands;
  * each rank's partial is the GEMM's bf16 output, summed in bf16 by the
    collective (the plainest reading of a psum over the bf16 dB); with P ranks
    a ring sum rounds P - 1 times;
  * the weight's rows are split evenly (N a multiple of the world size).

Overlap: `sharded_linear_backward` runs the wgrad GEMM first, starts the
reduce-scatter asynchronously (the collective's stream waits for the GEMM),
then runs the dgrad GEMM while the reduction is in flight, and waits only
before returning the dW shard.  Every cast and GEMM runs in the library's
kernels; the collective is torch.distributed's (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import gemm_fp4, gemm_fp4_bf16_wgrad

BLOCK = 32  # tokens per quantization block of the wgrad operands


def shard_rows(total: int, world: int, rank: int, multiple: int = BLOCK) -> tuple[int, int]:
    """[start, stop) of rank's contiguous shard of `total` rows: boundaries on
    multiples of `multiple` (total itself must be one), shards as even as that
    allows (the first total/multiple % world ranks get one block more)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if total % multiple:
        raise ValueError(f"{total} rows are not a multiple of {multiple}")
    blocks = total // multiple
    base, extra = divmod(blocks, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start * multiple, stop * multiple


def owned_rows(n: int, world: int, rank: int) -> tuple[int, int]:
    """[start, stop) of the dW rows rank receives from the reduce-scatter."""
    if n % world:
        raise ValueError(f"the weight's {n} rows do not split over {world} ranks")
    per = n // world
    return rank * per, (rank + 1) * per


def reduce_scatter_wgrad(partial: torch.Tensor, group=None, out: torch.Tensor | None = None,
                         async_op: bool = False):
    """Sum the ranks' partial dW [N, K] and keep this rank's rows.
    Returns (shard [N / P, K], work); work is None unless async_op."""
    world = dist.get_world_size(group)
    n = partial.shape[0]
    rows = owned_rows(n, world, dist.get_rank(group))
    if out is None:
        out = torch.empty((rows[1] - rows[0],) + tuple(partial.shape[1:]), dtype=partial.dtype,
                          device=partial.device)
    work = dist.reduce_scatter_tensor(out, partial.contiguous(), op=dist.ReduceOp.SUM, group=group,
                                      async_op=async_op)
    return out, work


def sharded_wgrad(dy: torch.Tensor, x: torch.Tensor, group=None, hadamard: bool = True) -> torch.Tensor:
    """This rank's rows of dW = sum_r dY_r^T X_r for bf16 token shards dY_r[M_r, N]
    and X_r[M_r, K] (M_r a multiple of 32): MXFP4 wgrad of the local tokens,
    then the reduce-scatter."""
    partial = gemm_fp4_bf16_wgrad(dy, x, hadamard=hadamard)
    shard, _ = reduce_scatter_wgrad(partial, group)
    return shard


def sharded_linear_backward(dy_q, x_q, w_q, group=None, stream=None):
    """Backward of y = x w^T on this rank's token shard, with the reduce-scatter
    of dW overlapped with the dgrad GEMM.

    dy_q: the grad preset's casts of the local dY[M_r, N] (row copy for dgrad,
          column copy with the Hadamard for wgrad), an MXFP4Tensor;
    x_q:  the activation preset's casts of the local X[M_r, K] (its column copy,
          with the Hadamard, is the wgrad operand);
    w_q:  the weight's casts (its column copy is the dgrad operand).
    Returns (dX_r [M_r, K] bf16, this rank's rows of dW [N / P, K] bf16)."""
    M, N = dy_q.rows, dy_q.cols
    K = x_q.cols
    if x_q.rows != M or w_q.rows != N or w_q.cols != K:
        raise ValueError("dy, x and w shapes do not form one linear layer")
    if dy_q.q_col is None or x_q.q_col is None:
        raise ValueError("the wgrad needs the column copies of dy and x")
    s = stream if stream is not None else torch.cuda.current_stream(dy_q.q_row.device)
    # dW_r[N, K] = dY_r^T . X_r: column copies, contraction over the local tokens
    partial = gemm_fp4(dy_q.q_col, dy_q.sf_col, x_q.q_col, x_q.sf_col, N, K, M, stream=s)
    with torch.cuda.stream(s):
        shard, work = reduce_scatter_wgrad(partial, group, async_op=True)
        # dX_r[M, K] = dY_r . W: row copy of dY against the column copy of W,
        # while the reduction is in flight
        dx = gemm_fp4(dy_q.q_row, dy_q.sf_row, w_q.q_col, w_q.sf_col, M, K, N, stream=s)
        work.wait()  # the stream waits for the collective
    return dx, shard
