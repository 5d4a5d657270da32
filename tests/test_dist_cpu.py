"""The N > 1 path of the benchmark on CPU: two gloo ranks.

Each rank owns its own slice of the global batch (weak scaling, no data-path
collective); the timed region's length is the max over ranks and the token
count the sum.  Checked with world_size 2 on the CPU (gloo, 127.0.0.1).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist = bench.dist_init(w, "gloo")
    wl = bench.build_workload("gqa4_b64", r, w, extra_steps=2)
    t_local = 1.0 + rank  # rank 1 is the slow one
    tmax = bench.reduce_max(t_local, dist, "cpu")
    tokens = bench.reduce_sum(float(wl.lengths.sum()), dist, "cpu")
    out[rank] = (wl.lengths.tolist(), tmax, tokens, wl.seed, wl.num_blocks)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharding_and_reductions():
    import synth
    import synth.workloads as W

    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    glob = synth.lengths_mix(synth.stream_seed(W.gqa4_b64().seed, W.TAG_LENGTHS), 64 * world)
    l0, tmax0, tok0, seed0, _ = out[0]
    l1, tmax1, tok1, seed1, _ = out[1]
    assert l0 == glob[:64].tolist() and l1 == glob[64:].tolist()  # disjoint shards of one draw
    assert l0 == W.gqa4_b64().lengths.tolist()  # rank 0 of N is the 1-GPU workload
    assert tmax0 == tmax1 == 2.0  # max over ranks
    assert tok0 == tok1 == float(glob.sum())  # whole-job token count
    assert seed0 != seed1  # independent data per rank


def test_shard_lengths_rejects_short_draw():
    import bench

    with pytest.raises(AssertionError):
        bench.shard_lengths(np.arange(10), 1, 2, 8)
