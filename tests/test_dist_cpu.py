"""The token-sharded wgrad with a reduce-scatter of dW (quantization_mxfp4_cast_gb300.dist)
on two gloo ranks, on CPU, with oracle partials: the library's sharding and
reduce-scatter bookkeeping against the unsharded oracle wgrad.

Method: jax-aiter README, "Supported ops" row "FP4 GEMM (training)" (FSDP-aware
wgrad sharding), "Quick start" (NT wgrad with FSDP-aware psum sharding).

Each rank takes its token shard (shard_rows: contiguous, on 32-token
boundaries), computes its partial dW_r = dY_r^T X_r with the oracle (column
casts with the Hadamard along its own tokens), rounds it to bf16 as the GEMM
does, and calls reduce_scatter_wgrad.  Bound, from the arithmetic: each
partial rounds once to bf16 and the two-term sum rounds once more, so
|got - dW| <= 2^-8 (|d_0| + |d_1| + |dW|) (1 + 2^-8) elementwise (2^-8: the unit
roundoff of bf16's 8-bit significand), with d_r the
exact partials and dW = d_0 + d_1 the unsharded oracle wgrad."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, N, K = 352, 64, 96  # 11 token blocks: uneven shards of 6 and 5 blocks


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def layer_inputs():
    from quantization_mxfp4_cast_gb300 import synth
    x = synth.normal_bf16((M, K), 1.0, seed=21)
    dy = synth.with_outliers(synth.normal_bf16((M, N), 1e-3, seed=22), frac=0.01)
    return x, dy


def oracle_wgrad(bx, bdy):
    import oracle
    ca, sa = oracle.cast_cols(np.ascontiguousarray(bdy), hadamard=True)
    cb, sb = oracle.cast_cols(np.ascontiguousarray(bx), hadamard=True)
    return oracle.gemm_mxfp4(ca, sa, cb, sb)


def worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from quantization_mxfp4_cast_gb300 import dist as mdist

    x, dy = layer_inputs()
    lo, hi = mdist.shard_rows(M, world, rank)
    part = oracle_wgrad(oracle.as_bf16_bits(x)[lo:hi], oracle.as_bf16_bits(dy)[lo:hi])
    np.save(os.path.join(out_dir, f"partial{rank}.npy"), part)
    shard, work = mdist.reduce_scatter_wgrad(torch.from_numpy(part).to(torch.bfloat16))
    assert work is None and shard.dtype == torch.bfloat16
    np.save(os.path.join(out_dir, f"shard{rank}.npy"), shard.float().numpy())
    dist.destroy_process_group()


def test_shard_boundaries():
    from quantization_mxfp4_cast_gb300.dist import owned_rows, shard_rows
    for total, world in ((352, 2), (8192, 8), (8192, 3), (96, 4), (32, 1)):
        bounds = [shard_rows(total, world, r) for r in range(world)]
        assert bounds[0][0] == 0 and bounds[-1][1] == total
        for (a, b), (c, _) in zip(bounds, bounds[1:]):
            assert b == c
        sizes = [b - a for a, b in bounds]
        assert all(s % 32 == 0 for s in sizes) and max(sizes) - min(sizes) <= 32
    assert [owned_rows(64, 4, r) for r in range(4)] == [(0, 16), (16, 32), (32, 48), (48, 64)]
    with pytest.raises(ValueError):
        shard_rows(100, 2, 0)
    with pytest.raises(ValueError):
        owned_rows(10, 4, 0)


def test_shard_casts_are_the_full_casts_split():
    # No 32-token block straddles a shard boundary, so the column casts (with
    # the Hadamard) of the shards are the full tensor's casts, split along the
    # tokens: sum_r dW_r is exactly the unsharded wgrad of the same operands.
    import oracle
    from quantization_mxfp4_cast_gb300.dist import shard_rows
    x, _ = layer_inputs()
    bx = oracle.as_bf16_bits(x)
    full_c, full_s = oracle.cast_cols(bx, hadamard=True)
    for r in range(2):
        lo, hi = shard_rows(M, 2, r)
        c, s = oracle.cast_cols(np.ascontiguousarray(bx[lo:hi]), hadamard=True)
        assert np.array_equal(c, full_c[:, lo // 2:hi // 2])
        assert np.array_equal(s, full_s[:, lo // 32:hi // 32])


def test_reduce_scatter_of_token_shard_partials(tmp_path):
    world = 2
    mp.spawn(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    import oracle
    from quantization_mxfp4_cast_gb300.dist import owned_rows
    x, dy = layer_inputs()
    full = oracle_wgrad(oracle.as_bf16_bits(x), oracle.as_bf16_bits(dy))
    d = [np.load(tmp_path / f"partial{r}.npy") for r in range(world)]
    assert np.allclose(d[0] + d[1], full, rtol=1e-12, atol=1e-14)  # exact partials sum to the whole
    bound = 2.0 ** -8 * (np.abs(d[0]) + np.abs(d[1]) + np.abs(full)) * (1 + 2.0 ** -8)
    for r in range(world):
        lo, hi = owned_rows(N, world, r)
        got = np.load(tmp_path / f"shard{r}.npy")
        assert got.shape == (hi - lo, K)
        assert np.all(np.abs(got - full[lo:hi]) <= bound[lo:hi]), f"rank {r}"
        # and it is the sum of the two bf16 partials, rounded once to bf16
        pb = [torch.from_numpy(q[lo:hi]).to(torch.bfloat16).float() for q in d]
        assert np.array_equal(got, (pb[0] + pb[1]).to(torch.bfloat16).float().numpy())
