"""The JSON line of bench.py's reference arm (the oracle timed on the host cores) for every
workload, and its behaviour under a two-process launch: rank 0 alone prints, every rank
exits 0.  Runs on the CPU; the GPU arm prints the same keys plus its roofline, clocks and
launch count, which only a GPU run can fill."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _run(args, timeout=240, env=None):
    return subprocess.run([sys.executable, *args], cwd=ROOT, capture_output=True, text=True, timeout=timeout,
                          env=env)


@pytest.mark.parametrize("workload", sorted(bench.WORKLOADS))
def test_reference_arm_prints_one_contract_line(workload):
    p = _run(["bench.py", "--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "0",
              "--all-core-budget", "1"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["name"] == workload and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["sample"] and cb["value"] == d["value"]
    ac = cb["all_core"]
    assert ac["cores"] == bench.host_cores() and ac["value"] > 0 and ac["unit"] == "tokens/s" and ac["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    p = _run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
              "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
              "--warmup", "0", "--workload", "hca_decode_1m", "--all-core-budget", "0"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
    assert "all_core" not in lines[0]["cpu_baseline"]


def test_all_core_timing_counts_units_over_wall_time():
    import threading
    import time
    done = []
    lock = threading.Lock()

    def unit():
        time.sleep(0.01)
        with lock:
            done.append(1)

    rate = bench.oracle_all_core(unit, 0.2, 4)
    # four threads of 10 ms units for 0.2 s: about 400 units/s, never more than the units run
    assert 150 < rate < 450 and len(done) >= 40


def test_clock_summary_median_and_reason_bits():
    c = bench.ClockSampler(0)
    c.max_mhz = 2032.0
    c.samples = [(1900.0, 0x4), (2000.0, 0), (1800.0, 0x8 | 0x4), (2032.0, 0x40)]
    s = c.summary()
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2032.0 and s["samples"] == 4
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples_says_why():
    c = bench.ClockSampler(0)
    c.error = "RuntimeError: NVML error 9"
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["error"] == c.error


def _traffic_rows():
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    rows = []
    for line in open(path).read().splitlines():
        cols = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cols) == 7 and cols[0] in bench.WORKLOADS:
            rows.append(cols)
    return rows


def test_traffic_table_rows_add_up():
    rows = _traffic_rows()
    assert rows
    for cols in rows:
        assert int(cols[4]) == int(cols[2]) + int(cols[3]), cols[0]


def test_traffic_counts_only_for_the_sources_it_was_taken_with(monkeypatch):
    rows = _traffic_rows()
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    assert all(bench.measured_traffic(w) is None for w in bench.WORKLOADS)
    name, h, traffic = rows[0][0], rows[0][6], int(rows[0][4])
    monkeypatch.setattr(bench, "source_hash", lambda: h)
    assert bench.measured_traffic(name) == traffic
