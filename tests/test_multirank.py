"""The N > 1 path of bench.py on CPU: two ranks over the gloo backend (the
GPU run uses NCCL; the host logic is the same). Checks that the ranks' input
shards are disjoint and together equal the single-process input stream, that
the job time is the slowest rank's, that the whole-job rate counts every
rank's evaluations, and that the reference arm runs on rank 0 only."""
import dataclasses
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    from mlp_neural_gb300 import synth

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        w = dataclasses.replace(synth.WORKLOADS["tiny"], n_unique=384)
        start, count = bench.rank_shard(w, rank)
        x = synth.inputs(w, start, count)
        assert x.shape == (count, w.dims[0])
        # gather every rank's shard on every rank; together they are the
        # first world * n_unique rows of the single-process stream
        parts = [torch.empty(count * w.dims[0], dtype=torch.int32) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(x.astype(np.int32).ravel()))
        joined = np.concatenate([p.numpy() for p in parts]).astype(np.uint16)
        whole = synth.inputs(w, 0, world * count)
        assert np.array_equal(joined, whole.ravel())
        # the job's time is the slowest rank's
        mine = 1.5 * (rank + 1)
        assert bench.max_over_ranks(mine, world, "cpu") == 1.5 * world
        # whole-job rate: every rank's evaluations over that time
        rate = bench.whole_job_rate(w.n_evals, 10, world, 1.5 * world)
        assert rate == pytest.approx(w.n_evals * 10 * world / (1.5 * world) / 1e6)
        # the reference arm: rank 0 only; the other ranks return at once
        if rank != 0:
            args = bench.parse_args(["--impl", "reference", "--gpus", str(world)])
            assert bench.run_reference(args, w, rank) == 0
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo():
    import torch.multiprocessing as mp
    mp.spawn(_worker, args=(2, _free_port()), nprocs=2, join=True)


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    from mlp_neural_gb300 import synth
    w = synth.WORKLOADS["page"]
    assert bench.rank_shard(w, 0) == (0, w.n_unique)
    assert bench.rank_shard(w, 3) == (3 * w.n_unique, w.n_unique)
