"""The bench's multi-rank host logic on two CPU processes (gloo): every rank gets a token shard
of the same shape with its own data, the job time is the slowest rank's, and throughput counts
every rank's tokens. The GR step itself has no collective (tokens are independent)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from stream_gated_residual_gb300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.shard(wl.WORKLOADS["tiny_fp32"], rank)
        R = wl.make_state(w)
        ms = bench.max_over_ranks(10.0 + rank, world)
        # a slowdown seen by one rank only: every rank decides to re-measure
        again = bench.any_over_ranks(rank == 1, world)
        neither = bench.any_over_ranks(False, world)
        tps = bench.job_tokens_per_s(world, w.n_tokens, 7, ms / 1e3)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), R=R, seed=w.seed, ms=ms, tps=tps,
                 again=again, neither=neither)
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_timing(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    base = wl.WORKLOADS["tiny_fp32"]
    assert [int(x["seed"]) for x in r] == [base.seed, base.seed + 1]
    assert r[0]["R"].shape == r[1]["R"].shape == (base.n_tokens, 4, base.d_model)
    assert not np.array_equal(r[0]["R"], r[1]["R"])          # different shards
    for x in r:
        assert float(x["ms"]) == 11.0                        # the slowest rank's time
        assert float(x["tps"]) == pytest.approx(world * base.n_tokens * 7 / 0.011)
        assert bool(x["again"]) is True and bool(x["neither"]) is False


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(1, 100, 10, 2.0) == 500.0
    assert bench.any_over_ranks(True, 1) is True and bench.any_over_ranks(False, 1) is False
