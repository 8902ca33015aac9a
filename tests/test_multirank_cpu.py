"""The multi-rank path's host logic on CPU, world size 2 over gloo.

Ranks shard rows/tokens with no data-path collective; RoPE takes global
positions, so a rank's token shard with its slice of positions reproduces the
single-process result exactly.  The job's time is the maximum over ranks.
(Gathering outputs to rank 0 below is only for checking.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

WORLD = 2
TOKENS_PER_RANK = 5


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import oracle
        import synth

        # weak scaling: each rank holds TOKENS_PER_RANK tokens of one sequence
        total = WORLD * TOKENS_PER_RANK
        q, k, wq, wk, _ = synth.qk_inputs(total, 3, 2, 32, 77, torch.bfloat16, torch.float32)
        lo = bench.weak_positions_start(TOKENS_PER_RANK, rank)
        hi = lo + TOKENS_PER_RANK
        pos = torch.arange(lo, hi, dtype=torch.int32)
        qo, ko, *_ = oracle.qk_norm_rope(synth.to_oracle(q[lo:hi]), synth.to_oracle(k[lo:hi]),
                                         synth.to_oracle(wq), synth.to_oracle(wk), pos.numpy())
        # strong split of a row count
        r_lo, r_hi = bench.shard_range(13, WORLD, rank)
        parts = [None] * WORLD if rank == 0 else None
        dist.gather_object((qo, ko, r_lo, r_hi), parts, dst=0)
        t = bench.max_over_ranks(1.5 + rank, dist)
        if rank == 0:
            full = oracle.qk_norm_rope(synth.to_oracle(q), synth.to_oracle(k), synth.to_oracle(wq),
                                       synth.to_oracle(wk), np.arange(total, dtype=np.int32))
            assert np.array_equal(np.concatenate([p[0] for p in parts]), full[0])
            assert np.array_equal(np.concatenate([p[1] for p in parts]), full[1])
            ranges = sorted((p[2], p[3]) for p in parts)
            assert ranges[0][0] == 0 and ranges[-1][1] == 13
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            assert t == 1.5 + WORLD - 1
            open(os.path.join(result_dir, "ok"), "w").write("ok")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_without_exchange(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=WORLD, join=True,
                       start_method="spawn")
    assert (tmp_path / "ok").exists()


@pytest.mark.parametrize("total,world", [(0, 2), (1, 2), (13, 2), (26598, 8), (7, 3)])
def test_shard_range_partitions(total, world):
    ranges = [bench.shard_range(total, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == total
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    sizes = [hi - lo for lo, hi in ranges]
    assert max(sizes) - min(sizes) <= 1
