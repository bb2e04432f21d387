"""The replica plumbing of bench.py on CPU: two gloo ranks, barrier and the
max over ranks that the timed region uses; the reference arm runs on rank 0
only and prints one contract line."""
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


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON
    line with the headline metric, its own cpu_baseline and a zero-copy e2e."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3 and d["config"]["workload"] == "long262k"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_cpu_baseline_on_one_and_on_several_cores():
    """The bench's CPU baseline: the oracle on one core and in one process per
    core (two here), with the cores, their model and both rates reported."""
    import bench
    from sparse_attention_indexer_kpool_gb300 import synth
    bt = synth.make_batch(synth.GEO_MAIN, [2048] * 4, [0] * 4, device="cpu", seed=5)
    bt.q_pos = None
    cb = bench.cpu_baseline((bt, bench.oracle_layer_cache(bt)), 0.3, cores=2)
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT
    assert cb["cores"] == cb["cores_all"] == 2
    assert cb["value"] == cb["value_all"] > 0 and cb["value_1core"] > 0
    assert isinstance(cb["cpu_model"], str) and cb["sample"]
