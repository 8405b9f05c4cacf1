"""The multi-rank host path of bench.py on CPU: two gloo ranks, each an independent replica.

Decode queries are independent, so ranks never exchange data: each rank draws its own batches
(different seeds), runs the chain on them (here the oracle stands in for the GPU kernels, since
this test runs without a GPU), and only the per-step time is reduced (maximum over ranks).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import synth

    wl = synth.small_workload("decode_b8_l32k_bf16", T=2, L=600, K=64)
    inputs = synth.make_inputs(wl, seed_offset=bench.rank_seed_offset(rank, 0))
    ch = oracle.Chain(synth.to_numpy_bits(inputs), L=wl.L, K=wl.K, q_per_seq=1, q_pos0=-1,
                      idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)
    r = oracle.chain_query(ch, 0, wl.D_v)
    ms = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
    first_idx = torch.tensor(r["idx"][:8].astype(np.int64))
    gathered = [torch.zeros_like(first_idx) for _ in range(world)]
    dist.all_gather(gathered, first_idx)  # test-only check that the replicas drew different data
    out[rank] = (ms, [g.tolist() for g in gathered], bench.rank_seed_offset(rank, 0))
    dist.destroy_process_group()


def test_two_gloo_ranks_run_independent_replicas_and_reduce_the_slowest_time():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 2.0          # max over ranks of (1.0, 2.0)
    assert out[0][2] != out[1][2]                  # distinct seeds per rank
    assert out[0][1][0] != out[0][1][1]            # the two replicas scored different data
