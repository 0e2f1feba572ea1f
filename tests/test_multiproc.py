"""Host logic of the multi-GPU bench path, run as two gloo ranks on the CPU.

The decode step shards by sequence with no collective on the data path; the
only cross-rank steps are the barrier and the max / sum reductions of the
timing. Those, and the row split, are exercised here without a GPU.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rows = bench.shard_rows(rank, 64)
        mx = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        sm = bench.sum_over_ranks(100.0 * (rank + 1), world, torch.device("cpu"))
        bench.barrier(world)
        out[rank] = (rows, mx, sm)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_reduce_timings():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == (0, 64) and out[1][0] == (64, 128)
    assert out[0][1] == out[1][1] == 2.5       # the slowest rank's time
    assert out[0][2] == out[1][2] == 300.0     # total updates over ranks


def test_rank_shards_are_disjoint_slices_of_the_global_batch():
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=4, L=2)
    whole = W.sequence_slice(w, 3, 1)
    # rank 1 of 2 with 2 rows per rank owns global sequences 2 and 3
    b0, b1 = bench.shard_rows(1, 2)
    assert (b0, b1) == (2, 4)
    assert np.array_equal(W.sequence_slice(w, b1 - 1, 1)["state"], whole["state"])


def test_counting_of_updates_and_algorithmic_bytes():
    w = W.WORKLOADS["decode_b64_l36_t1"]
    assert bench.valid_tokens(w, None) == 64 * 36
    b = bench.algorithmic_bytes(w, None)
    assert b["state"] == 64 * 36 * 48 * 65536 * 2
    assert b["total"] == 15276178944
    r = W.WORKLOADS["verify_b16_l36_t8_ragged"]
    lens = W.seq_lens(r)
    assert bench.valid_tokens(r, lens) == int(lens.sum()) * 36
