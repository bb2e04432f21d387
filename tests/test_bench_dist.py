"""The replica plumbing of bench.py on CPU: two gloo ranks, barrier and the
max over ranks that the timed region uses; the reference arm runs on rank 0
only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist(world)
    try:
        d.barrier()
        m = d.max(10.0 + rank)                     # each rank's own time
        class Args:                                # a reference-arm call on every rank
            steps, warmup, seqlen = 1, 0, 4096
        printed = []
        if rank != 0:
            bench.run_reference(Args, d)           # must return at once, printing nothing
            printed.append("returned")
        d.barrier()
    finally:
        d.close()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{d.world} {d.rank} {m} {' '.join(printed)}")


def test_two_gloo_ranks_take_the_max(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r0 = open(tmp_path / "rank0.txt").read().split()
    r1 = open(tmp_path / "rank1.txt").read().split()
    assert r0[:3] == ["2", "0", "11.0"] and r1[:3] == ["2", "1", "11.0"]
    assert r1[3:] == ["returned"]


def test_single_process_needs_no_process_group():
    import bench
    for k in ("WORLD_SIZE", "RANK"):
        assert k not in os.environ or os.environ[k] in ("1", "0")
    d = bench.Dist(1)
    assert d.pg is None and d.max(3.5) == 3.5
    d.barrier()
    d.close()
