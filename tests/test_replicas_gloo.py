"""Multi-process host logic of the replica bench, on CPU ranks (gloo).

Each rank runs an independent replica of the output stage (no sharding, no
collective): `bench.py --gpus N` runs N of them and reports every rank's bytes
over the slowest rank's time.  These tests run that aggregation with two gloo ranks, and check that
the reference arm does its work on rank 0 only.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (1 + r) ms for 1e9 bytes: the job moved world * 1e9 bytes in max = world ms
        value, secs = bench.replica_aggregate((1.0 + rank) * 1e-3, 10**9)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{value!r} {secs!r}\n")
    finally:
        dist.destroy_process_group()


def test_replica_aggregate_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        value, secs = map(float, (tmp_path / f"r{r}.txt").read_text().split())
        assert secs == pytest.approx(2e-3)                     # the slowest rank's time on every rank
        assert value == pytest.approx(world * 1e9 / 2e-3 / 1e9)   # all ranks' bytes over it


def test_replica_aggregate_single_process_is_identity():
    import bench
    value, secs = bench.replica_aggregate(0.5, 10**9)
    assert secs == 0.5 and value == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse
    import bench
    import q5k_synth as synth
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args, synth.WORKLOADS["tiny"]) is None
    assert capsys.readouterr().out == ""                        # no line, no work on rank 1
