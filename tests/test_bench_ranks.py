"""bench.py's multi-rank logic on the CPU: two gloo ranks, each timing its
own replica; the job reports the slowest rank's times and N x the bytes."""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured step 1.0 + r ms, forward 0.3 + r, backward 0.7
        got = bench.slowest_rank(dist, [1.0 + rank, 0.3 + rank, 0.7], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_over_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        results = dict(out)
    assert set(results) == {0, 1}
    for rank in range(world):
        assert results[rank] == pytest.approx([2.0, 1.3, 0.7])


def test_replica_throughput_is_whole_job():
    one = bench.replica_throughput(1, 10**9, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.replica_throughput(4, 10**9, 1.0) == pytest.approx(4 * one)
    assert bench.slowest_rank(None, [1, 2.5], "cpu") == [1.0, 2.5]


def test_dist_env_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    monkeypatch.setenv("WORLD_SIZE", "8")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "3")
    assert bench.dist_env() == (3, 8, 3)


def test_cpu_baseline_reports_one_thread_and_all_cores():
    from memory_bound_normalization_gb300 import synth

    wl = synth.WORKLOADS["small_256x1024"]
    got = bench.cpu_baseline(wl, 0.2)
    assert got["kind"] == "oracle" and got["cores"] == 1 and got["value"] > 0
    cores = os.cpu_count() or 1
    if cores > 1:
        allc = got["all_cores"]
        assert allc["cores"] == cores and allc["value"] > 0 and allc["unit"] == got["unit"]


def test_reference_arm_prints_the_contract_line(capsys):
    """bench.py --impl reference: the fp64 oracle on the host cores, one JSON
    line with the keys the contract names (small budget here)."""
    import json

    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--ref-seconds", "0.3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["metric"] and line["config"]["workload"]


def test_profiled_traffic_only_for_the_current_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary of the backward
    only while that summary's source hash is the one given (the current
    sources'); a missing summary or another hash gives None."""
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "rmsnorm_bwd_wl.md").write_text(
        "# summary\n\nsource_hash: 0123456789abcdef\n\ntraffic_bytes_per_launch: 354168064\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_profiled_traffic("rmsnorm_bwd", "wl", "0123456789abcdef") == 354168064
    assert bench.read_profiled_traffic("rmsnorm_bwd", "wl", "fedcba9876543210") is None
    assert bench.read_profiled_traffic("rmsnorm_bwd", "other", "0123456789abcdef") is None
