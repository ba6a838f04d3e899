"""Multi-process paths on CPU (gloo, world size 2).

A multi-GPU run shards the decode batch: every rank decodes its own sequences,
and the only collective is the maximum of the ranks' step times.  These tests
run that host logic as two gloo ranks on the CPU:
  * ``bench.max_over_ranks`` gives every rank the largest value;
  * decoding a batch as two shards of sequences, one per rank, gives exactly
    the results of decoding it in one process (the float64 oracle: sequences
    share nothing, so no exchange is needed).
"""
from __future__ import annotations

import dataclasses
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import synth

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank: int, port: int):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    return dist


def _max_worker(rank: int, port: int):
    dist = _init(rank, port)
    import bench
    got = bench.max_over_ranks(10.0 + 3.0 * rank, device="cpu")
    assert got == 10.0 + 3.0 * (WORLD - 1), got
    dist.destroy_process_group()


def _small_decode():
    return synth.Workload("shard", "decode", B=4, L=4100, T=1, R=128, k=64, W=32, m2=16,
                          x8=True)


def _shard(w, x, lo, hi):
    sub = dataclasses.replace(w, B=hi - lo)
    xs = {k: (v[lo:hi] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == w.B
              else v) for k, v in x.items()}
    return sub, xs


def _shard_worker(rank: int, port: int):
    dist = _init(rank, port)
    w = _small_decode()
    x = synth.make_inputs(w)
    per = w.B // WORLD
    sub, xs = _shard(w, x, rank * per, (rank + 1) * per)
    mine = oracle.reference(sub, xs)
    parts = [None] * WORLD
    dist.all_gather_object(parts, {k: mine[k] for k in ("idx", "o", "lse", "ho", "hlse")})
    if rank == 0:
        full = oracle.reference(w, x)
        for k in ("idx", "o", "lse", "ho", "hlse"):
            joined = np.concatenate([p[k] for p in parts], axis=0)
            assert joined.shape == full[k].shape, (k, joined.shape, full[k].shape)
            np.testing.assert_array_equal(joined, full[k], err_msg=k)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_max_over_ranks_gloo():
    mp.spawn(_max_worker, args=(_free_port(),), nprocs=WORLD, join=True)


@pytest.mark.timeout(600)
def test_batch_shards_equal_one_process_gloo():
    mp.spawn(_shard_worker, args=(_free_port(),), nprocs=WORLD, join=True)
