"""The N > 1 bench path on the CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own replica of the workload (weak scaling); the only collective is
the max-over-ranks of the step time (not on the data path) and a barrier.  This checks
the rank plumbing, the max reduction and the whole-job value arithmetic with world
size 2, and that each rank draws the identical seeded workload.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from paged_gqa_attention_gb300 import workloads as wl

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    # per-rank "step times": the job time is the slowest rank's
    step_ms = 1.0 + rank
    job_ms = bench.dist_max(step_ms, w)
    bench.dist_barrier(w)
    # each rank's replica is the same seeded workload (weak scaling: work per rank fixed)
    b = wl.build_batch("replica", 7, [300, 40, 513], [1, 1, 1], num_blocks=8)
    digest = float(b.q.float().sum() + b.k_pool.float().nan_to_num().sum())
    kv = b.kv_bytes()
    value = w * kv / (job_ms * 1e-3) / 1e9
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{job_ms} {digest} {value} {kv}\n")
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_share_the_workload(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    job = [float(x[0]) for x in rows]
    digests = [float(x[1]) for x in rows]
    values = [float(x[2]) for x in rows]
    kv = int(rows[0][3])
    assert job == [2.0, 2.0]                      # max over ranks seen by every rank
    assert digests[0] == digests[1]               # identical seeded replica on each rank
    assert values[0] == pytest.approx(world * kv / 2e-3 / 1e9)
