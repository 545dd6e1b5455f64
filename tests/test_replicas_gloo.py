"""The N > 1 path on CPU: two gloo ranks compute column shards of one GEMM with
the oracle, gather them, and must reproduce the single-rank result bit for bit;
the max-over-ranks timing and the whole-job rate are checked on the same ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from roofline_driven_optimisation_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from roofline_driven_optimisation_gb300 import inputs
        c = inputs.make("fp32_4096", M=24, N=37, K=19)
        n0, n1 = replicas.column_shard(37, world, rank)
        part = oracle.gemm(c.A, c.B[:, n0:n1], 1.5, 0.5, c.C0[:, n0:n1], threads=1)
        shards = [None] * world
        dist.all_gather_object(shards, (n0, n1, part))
        t = replicas.max_over_ranks(1.5 + rank, dist)
        rate = replicas.whole_job_rate(10.0, world, t)
        if rank == 0:
            full = np.concatenate([s[2] for s in sorted(shards, key=lambda s: s[0])], axis=1)
            np.save(os.path.join(out_dir, "gathered.npy"), full)
            with open(os.path.join(out_dir, "timing.txt"), "w") as f:
                f.write(f"{t} {rate}\n")
    finally:
        dist.destroy_process_group()


def test_column_shards_cover_exactly():
    for n in (0, 1, 5, 37, 4096):
        for world in (1, 2, 3, 8):
            spans = [replicas.column_shard(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            widths = [b - a for a, b in spans]
            assert max(widths) - min(widths) <= 1
    with pytest.raises(ValueError):
        replicas.column_shard(4, 2, 2)


def test_single_process_fallbacks():
    assert replicas.max_over_ranks(3.25) == 3.25
    assert replicas.whole_job_rate(6.0, 4, 2.0) == 12.0


def test_two_gloo_ranks_reproduce_the_full_gemm(tmp_path):
    import oracle
    from roofline_driven_optimisation_gb300 import inputs
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    c = inputs.make("fp32_4096", M=24, N=37, K=19)
    want = oracle.gemm(c.A, c.B, 1.5, 0.5, c.C0, threads=1)
    got = np.load(tmp_path / "gathered.npy")
    assert np.array_equal(got, want)
    t, rate = map(float, open(tmp_path / "timing.txt").read().split())
    assert t == 2.5                      # the slower rank's time
    assert rate == world * 10.0 / 2.5    # every rank's work over that time
