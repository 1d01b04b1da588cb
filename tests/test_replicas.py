"""The N > 1 path of bench.py on CPU: world-size-2 gloo process groups.

The decode path does not shard: N GPUs run N independent replicas, joined only
by a barrier around the timed region and the max over ranks of its time. These
tests run that host logic as two gloo ranks on 127.0.0.1 (no GPU).
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch
    import bench
    dist = bench.replica_group("gloo")
    assert dist is not None and dist.get_world_size() == world
    dist.barrier()
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slower replica
    ms = bench.max_over_ranks(torch, ms_local, "cpu", dist)
    value = bench.job_value(2_000_000, 100, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "ws": bench.dist_info()[0]}, f)


def test_two_gloo_replicas_agree_on_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["ws"] == world
        assert r["ms"] == 15.0                               # max over ranks, on every rank
        # whole job: 2 replicas x 100 steps x 2 MB in 15 ms
        assert r["value"] == pytest.approx(2 * 100 * 2_000_000 / 15e-3 / 1e9)


def test_single_process_needs_no_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_info() == (1, 0, 0)
    assert bench.replica_group("gloo") is None
    assert bench.max_over_ranks(None, 3.5, "cpu", None) == 3.5
    assert bench.job_value(1e9, 10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 3, "warmup": 3, "gpus": 2})()
    assert bench.run_reference(args) == 0   # returns at once, without work
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_0(monkeypatch, capsys):
    """Rank 0 (or a single process) times the oracle on a bounded sample and
    prints one JSON line with the keys of the benchmark contract: the
    reference tag, the metric and unit of the GPU line, a cpu_baseline
    block describing the run, and an e2e block with no host-device copies."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    oracle.build()
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    args = type("A", (), {"steps": 1, "warmup": 3, "gpus": 1})()
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    for key in ("value", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
                "dtype", "data", "config"):
        assert key in line, key
    assert line["value"] > 0 and line["higher_is_better"] is True and line["config"]["workload"] == "decode_2b"
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"] and cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
