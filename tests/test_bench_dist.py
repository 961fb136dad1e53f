"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each an
independent replica; the step time is the slowest rank's and the whole-job
value counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = 2.0 + 3.0 * rank          # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, world)
        out[rank] = ms_max
        out[world + rank] = bench.replica_gbs(1_000_000, world, ms_max)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    world = 2
    out = mp.get_context("spawn").Array("d", 2 * world)
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert list(out[:world]) == [5.0, 5.0]
    # 2 replicas x 1 MB in 5 ms = 0.4 GB/s, the same on every rank
    assert out[world:] == pytest.approx([0.4, 0.4])


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_gbs(2_000_000_000, 1, 1000.0) == pytest.approx(2.0)


def test_attention_flop_count_matches_brute_force():
    """bench.attn_flops: 4 * D flops per (visible token, query head), position j
    of a sequence with context L seeing L - T + 1 + j tokens."""
    import dataclasses
    import bench
    from bit_kv_cache_rotate_b300 import workloads as W
    cfg = dataclasses.replace(W.CONFIGS["extend_b4_ctx32k_t512"], q_per_seq=5, num_q_heads=6, head_dim=64)
    lens = [5, 9, 40]
    brute = sum(4 * 64 * 6 * (L - 5 + 1 + j) for L in lens for j in range(5))
    assert bench.attn_flops(cfg, lens) == brute
    assert bench.is_extend(cfg) is False
    assert bench.is_extend(W.CONFIGS["extend_b4_ctx32k_t512"]) is True
