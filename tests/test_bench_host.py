"""CPU checks of bench.py's host logic: the clock-sample summary, the profile-traffic
lookup gated by the kernel's source hash, and the synthetic workloads' shapes."""
import os
import shutil

import numpy as np

import bench
from stream_compaction_decoupled_gb300 import workloads


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def _line(ts, sm, mx, hw="Not Active", sw_power="Not Active"):
    return "%s, 0, %d, %d, 900.0, 0x0, %s, Not Active, Not Active, %s" % (ts, sm, mx, hw, sw_power)


def test_clock_summary_inside_the_timed_region(tmp_path):
    import datetime as dt
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line((t0 + dt.timedelta(seconds=0.1 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3],
                   2070 if i != 3 else 1900, 2070, sw_power="Active" if i == 4 else "Not Active")
             for i in range(10)]
    s = _sampler_with(tmp_path, lines)
    a, b = t0.timestamp() + 0.15, t0.timestamp() + 0.55
    out = s.summary(a, b)
    assert out["window"] == "timed region" and out["samples"] == 4
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_hw_slowdown_and_short_regions(tmp_path):
    import datetime as dt
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line((t0 + dt.timedelta(seconds=0.1 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], 1500, 2070,
                   hw="Active") for i in range(5)]
    s = _sampler_with(tmp_path, lines)
    x = t0.timestamp() + 0.42  # shorter than the sampling period: falls back to the load around it
    out = s.summary(x, x + 0.01)
    assert out["reasons"] == ["hw_slowdown"] and out["samples"] >= 1
    assert out["window"].startswith("benchmark load")
    empty = _sampler_with(tmp_path, [])
    assert empty.summary(0, 1)["samples"] == 0


def test_profile_traffic_needs_the_current_source_hash(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "stream_compaction_decoupled_gb300", "csrc"),
                    root / "stream_compaction_decoupled_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_source_hash("scan_stash_kernel")
    (root / "profiles" / "a.md").write_text(
        "kernel: scan_stash_kernel<float,add>\nsource_hash: %s\ntraffic_bytes_per_launch: 123456\n" % h)
    assert bench.traffic_from_profiles("scan_stash_kernel<float,add>") == 123456.0
    assert bench.traffic_from_profiles("scan_seg_kernel<float,add>") is None
    # editing one of the kernel's sources changes the hash and retires the figure
    f = root / "stream_compaction_decoupled_gb300" / "csrc" / "scan_stash.cuh"
    f.write_text(f.read_text() + "\n// edit\n")
    assert bench.kernel_source_hash("scan_stash_kernel") != h
    assert bench.traffic_from_profiles("scan_stash_kernel<float,add>") is None


def test_workload_shapes_and_seeds():
    for w in workloads.WORKLOADS:
        if w.elems * w.lanes > 30_000_000:  # the 1e8 headline arrays: shape by arithmetic only
            assert w.elems == 100_000_000
            continue
        x = w.make()
        assert x.size == w.elems * w.lanes, w.name
        assert x.dtype == np.dtype(w.dtype if w.kind != "pack" else np.int32), w.name
        assert np.array_equal(x[:1000], w.make()[:1000]), w.name  # seeded: the same bytes every time
    assert workloads.BY_NAME[workloads.HEADLINE].dtype == "float32"
    f = workloads.head_flags(100_000, 0.01, 3)
    assert f.dtype == np.uint8 and 500 < int(f.sum()) < 1500
