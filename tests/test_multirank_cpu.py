"""Two-rank (gloo, CPU) checks of the data-parallel structure of the path.

The casts and the forward / dgrad GEMMs split along the token dimension M with
no exchange; wgrad (dW = dY^T X, contraction over M) splits into per-shard
partials that sum to the whole (the README's "FSDP-aware wgrad" psum, jax-aiter
README "Supported ops" FP4 GEMM row).  With shards that are whole multiples of
the 32-token quantization (and Hadamard) block, every block is quantized
identically on its shard, so the summed partials equal the unsharded oracle
result up to fp64 summation order.  Also checks bench.py's max-over-ranks
timing helper."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from quantization_mxfp4_cast_gb300 import synth

    M, N, K = 256, 48, 64
    x, _, dy = synth.linear_layer(M, 32, K, x_sigma=1.0)
    dy = synth.normal_bf16((M, N), 1e-3, synth.SEED_DY)
    shard = M // world  # a multiple of 32 tokens
    lo, hi = rank * shard, (rank + 1) * shard
    bx = oracle.as_bf16_bits(x)[lo:hi]
    bdy = oracle.as_bf16_bits(dy)[lo:hi]
    ca, sa = oracle.cast_cols(np.ascontiguousarray(bdy), hadamard=True)
    cb, sb = oracle.cast_cols(np.ascontiguousarray(bx), hadamard=True)
    part = torch.from_numpy(oracle.gemm_mxfp4(ca, sa, cb, sb))
    dist.all_reduce(part, op=dist.ReduceOp.SUM)

    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    t_max = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
    bench.barrier(world)
    if rank == 0:
        np.save(os.path.join(out_dir, "summed.npy"), part.numpy())
        np.save(os.path.join(out_dir, "tmax.npy"), np.array([t_max]))
    dist.destroy_process_group()


def test_wgrad_token_shards_sum_to_the_whole(tmp_path):
    world = 2
    mp.spawn(worker, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    summed = np.load(tmp_path / "summed.npy")
    import oracle
    from quantization_mxfp4_cast_gb300 import synth
    M, N, K = 256, 48, 64
    x, _, _ = synth.linear_layer(M, 32, K, x_sigma=1.0)
    dy = synth.normal_bf16((M, N), 1e-3, synth.SEED_DY)
    ca, sa = oracle.cast_cols(oracle.as_bf16_bits(dy), hadamard=True)
    cb, sb = oracle.cast_cols(oracle.as_bf16_bits(x), hadamard=True)
    full = oracle.gemm_mxfp4(ca, sa, cb, sb)
    assert summed.shape == (N, K)
    assert np.allclose(summed, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())
    assert float(np.load(tmp_path / "tmax.npy")[0]) == float(world)
