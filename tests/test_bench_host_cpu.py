"""Host-side logic of bench.py on CPU (no GPU): the clock summary and the rule that
rejects a throttled or clock-locked run, and the workload table's generators."""
import os
import tempfile

import numpy as np
import pytest

import bench


def summary_of(lines):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = object()  # as if nvidia-smi had been started
    return s.summary()


def row(sm, smax, watts, hw="Not Active", hw_th="Not Active", sw_th="Not Active",
        cap="Not Active"):
    return f"0, {sm}, {smax}, {watts}, 0x0, {hw}, {hw_th}, {sw_th}, {cap}"


def test_clock_summary_uses_loaded_samples():
    s = summary_of([row(1000, 2070, 90.0), row(2070, 2070, 900.0), row(2070, 2070, 950.0),
                    row(2055, 2070, 940.0), "garbage line", "0, [N/A], 2070, 1, x, a, b, c, d"])
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 4
    assert s["reasons"] == [] and not bench.clocks_rejected(s)


@pytest.mark.parametrize("kw,rejected", [
    ({"hw": "Active"}, True), ({"hw_th": "Active"}, True), ({"sw_th": "Active"}, True),
    ({"cap": "Active"}, False)])
def test_throttle_reasons(kw, rejected):
    s = summary_of([row(2070, 2070, 900.0), row(1900, 2070, 1400.0, **kw)])
    assert bench.clocks_rejected(s) is rejected


def test_clock_lock_without_reason_is_rejected():
    locked = summary_of([row(900, 2070, 800.0), row(900, 2070, 810.0)])
    assert bench.clocks_rejected(locked)
    capped = summary_of([row(900, 2070, 1400.0, cap="Active")] * 2)
    assert not bench.clocks_rejected(capped)
    assert not bench.clocks_rejected(None)


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_workload_generators(name):
    """Every workload's prefix table and index sampler give valid shapes and rows."""
    wl = bench.workload_table(name)
    rows = wl["rows_prefix"](64)
    assert rows.ndim == 2 and rows.shape[0] == 64
    assert rows.shape[1] * rows.dtype.itemsize % 16 == 0
    idx = wl["index"](64, 200, 3)
    assert idx.dtype == np.int64 and idx.size == 200
    assert idx.min() >= 0 and idx.max() < 64
    assert wl["T"] in (0.9, 0.95) and wl["B"] in (32, 64) and wl["residency"] in ("host", "device")


def test_oracle_baselines_single_and_all_cores():
    """The cpu_baseline legs: the oracle single-threaded and split over every core,
    on a small prefix table and short budgets."""
    wl = bench.workload_table("tiny")
    one, every = bench.oracle_sample(wl, seconds_budget=0.2, sample_rows=2048,
                                     all_cores_budget=0.2)
    assert one["cores"] == 1 and every["cores"] == (os.cpu_count() or 1)
    for d in (one, every):
        assert d["kind"] == "oracle" and d["unit"] == "GB/s" and d["value"] > 0
        assert d["batches"] >= 1


def test_unknown_legs_are_refused_before_any_work():
    import subprocess
    import sys
    r = subprocess.run([sys.executable, bench.__file__, "--legs", "dedup,nonsense"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "unknown legs" in r.stderr and "nonsense" in r.stderr
