"""bench.py's host-side rules without a GPU: the idle-GPU verdict, the index
nvidia-smi is asked about, and the drift flag's threshold."""
from __future__ import annotations

import bench


def test_idle_verdict():
    assert bench.assess_idle([]) == {"checked": False, "busy": None}
    idle = bench.assess_idle([(0.0, 0.0), (3.0, 0.0), (0.0, 1.0)])
    assert idle["checked"] and idle["busy"] is False
    assert idle["memory_used_mib_max"] == 3.0 and idle["utilization_pct_max"] == 1.0
    # another process's memory, or work on the GPU, in any sample makes it busy
    assert bench.assess_idle([(0.0, 0.0), (bench.IDLE_MAX_MIB + 1.0, 0.0)])["busy"] is True
    assert bench.assess_idle([(0.0, bench.IDLE_MAX_UTIL + 1.0)])["busy"] is True
    assert bench.assess_idle([(bench.IDLE_MAX_MIB, bench.IDLE_MAX_UTIL)])["busy"] is False


def test_smi_index_follows_visible_devices(monkeypatch):
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    assert bench.smi_index(0) == "0" and bench.smi_index(3) == "3"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5,2")
    assert bench.smi_index(0) == "5" and bench.smi_index(1) == "2"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-1234abcd")
    assert bench.smi_index(0) == "0"


def test_drift_limit_and_new_options():
    assert bench.DRIFT_LIMIT == 0.98
    a = bench.parse_args([])
    assert a.probe_gib >= 4 and a.probe_samples >= 20
    assert a.steady_steps > 0 and not a.no_configs and not a.require_idle
    assert set(bench.CONFIG_WORKLOADS) == {"small_256x1024", "hidden8192_32768x8192_outliers",
                                           "qknorm_1048576x128"}


def test_statistics_helpers():
    xs = [float(v) for v in range(1, 11)]
    assert bench.p90(xs) == 9.0
    assert bench.p90([3.0]) == 3.0
    # step k runs on clone set k % nsets
    assert bench.by_set([1.0, 10.0, 3.0, 30.0, 5.0], 2) == [3.0, 20.0]
    assert bench.by_set([2.0, 4.0], 3) == [2.0, 4.0]


def test_steady_fields():
    assert bench.steady_fields({"steady": None}, 10**9, 1000.0) == {}
    got = bench.steady_fields({"steady": {"step_ms": 0.5}}, 10**9, 4000.0)
    assert got == {"steady_gbs": 2000.0, "steady_frac": 0.5}


def test_results_log_resume(tmp_path):
    d = str(tmp_path / "run")
    log = bench.ResultsLog(d)
    log.env({"gpu": "x"})
    log.add("sweep", {"workload": "a", "fwd_frac": 1.0})
    log.add("config", {"workload": "b", "bwd_frac": 0.9})
    with open(tmp_path / "run" / "cells.jsonl", "a") as f:
        f.write('{"kind": "sweep", "workload": "c", "fwd')  # cut off by an interruption
    again = bench.ResultsLog(d, resume=True)
    assert again.done("sweep", "a") == {"workload": "a", "fwd_frac": 1.0}
    assert again.done("config", "b") == {"workload": "b", "bwd_frac": 0.9}
    assert again.done("sweep", "c") is None and again.done("sweep", "b") is None
    fresh = bench.ResultsLog(d)  # without --resume the old cells are dropped
    assert fresh.done("sweep", "a") is None
    assert not (tmp_path / "run" / "cells.jsonl").exists()
    assert (tmp_path / "run" / "env.json").exists()
    assert bench.ResultsLog(None).done("sweep", "a") is None
