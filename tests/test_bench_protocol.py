"""bench.py's timing protocol as host logic (no GPU): rotating input/output
sets for the cold lane, batches of launches between events, median-based
statistics, the shared config of both arms and the row sample of the parity
gate."""
import numpy as np
import pytest

import bench
import synth


def test_rotation_reaches_the_rotation_bytes():
    for set_bytes in (1, 2 << 20, 134217728, 67108864 + 65536000, 1 << 30, 4294967296):
        r = bench.rotation_count(set_bytes, "cold")
        assert r * set_bytes >= bench.ROTATE_BYTES
        assert (r - 1) * set_bytes < bench.ROTATE_BYTES or r == 1
    assert bench.rotation_count(1 << 20, "warm") == 1
    # 4x a 129 MB L2 is inside the rotation span
    assert bench.ROTATE_BYTES >= 4 * 129_000_000


def test_headline_workloads_rotation():
    # The largest workload needs one set; the f32 4096^2 matrix needs 8 of 134 MB.
    c5 = synth.WORKLOADS["f16_causal_524288x2048"]
    c2 = synth.WORKLOADS["f32_4096x4096"]
    assert bench.rotation_count(2 * c5.M * c5.N * 2, "cold") == 1
    assert bench.rotation_count(2 * c2.M * c2.N * 4, "cold") == 8


def test_batch_plan():
    # ~200 us per batch, at least five batches when steps allow
    assert bench.batch_plan(20, 600.0) == 1
    assert bench.batch_plan(200, 12.0) == 17
    assert bench.batch_plan(20, 12.0) == 4
    assert bench.batch_plan(3, 12.0) == 3
    assert bench.batch_plan(1, 0.0) == 1
    for steps in (1, 2, 5, 7, 20, 100, 1000):
        for est in (0.5, 6.0, 20.0, 80.0, 600.0):
            b = bench.batch_plan(steps, est)
            assert 1 <= b <= steps
            if steps >= bench.MIN_BATCHES:
                assert steps // b >= bench.MIN_BATCHES


def test_batch_bounds_cover_every_step_once():
    for steps in (1, 5, 20, 21, 100):
        for b in (1, 3, 4, 17, 100):
            bounds = bench.batch_bounds(steps, b)
            covered = [k for s, e in bounds for k in range(s, e)]
            assert covered == list(range(steps))
            assert all(e - s == b for s, e in bounds[:-1])


def test_batch_stats_median_over_full_batches():
    bounds = bench.batch_bounds(10, 3)  # 3, 3, 3, 1
    batch_ms = [0.030, 0.036, 0.033, 0.100]  # the short last batch is an outlier
    st = bench.batch_stats(batch_ms, bounds)
    assert st["median_step_us"] == pytest.approx(11.0)
    assert st["mean_step_us"] == pytest.approx(sum(batch_ms) * 1e3 / 10)
    assert st["min_max_step_us"] == [pytest.approx(10.0), pytest.approx(12.0)]
    assert st["launches_per_batch"] == 3 and st["batches"] == 4
    # all batches short (one step): every batch counts
    st = bench.batch_stats([0.002], [(0, 1)])
    assert st["median_step_us"] == pytest.approx(2.0)


def test_both_arms_print_the_same_config():
    for w in synth.WORKLOADS.values():
        a = bench.workload_config(w, "cold", 1)
        b = bench.workload_config(w, "cold", 1)
        assert a == b
        assert set(a) == {"workload", "M", "N", "ld_in", "ld_out", "l2", "parallelism"}
    c5 = bench.workload_config(synth.WORKLOADS["f16_causal_524288x2048"], "cold", 1)
    assert c5["l2"].startswith("inputs larger than L2")
    c2 = bench.workload_config(synth.WORKLOADS["f32_4096x4096"], "cold", 1)
    assert c2["l2"].startswith("rotation: 8 input/output sets")


def test_parity_rows():
    assert list(bench.parity_rows(100, 1000)) == list(range(100))
    rows = bench.parity_rows(524288, 2048)
    assert rows[0] == 0 and rows[-1] == 524287
    assert len(rows) == (1 << 25) // 2048
    assert np.all(np.diff(rows) > 0)
    # the sample reaches many query positions of the causal period
    assert len(np.unique(rows % 2048)) > 1500
    assert np.array_equal(rows, bench.parity_rows(524288, 2048))  # seeded


def test_compare_rows_counts_planted_errors():
    w = synth.WORKLOADS["bf16_16384x1000_ld1024"].with_rows(4)
    rows = np.arange(4)
    ref = np.full((4, w.ld_out), 0x3C00, dtype=np.uint16)  # bf16 0.0078125
    got = ref.copy()
    assert bench.compare_rows(w, got, ref, rows)["outside_tolerance"] == 0
    got[2, 5] = 0x3F80  # 1.0
    got[3, 999] = 0x7FC0  # NaN where the oracle is finite
    r = bench.compare_rows(w, got, ref, rows)
    assert r["outside_tolerance"] == 2
    ref[1, 0] = got[1, 0] = 0x7FC0  # NaN on both sides passes
    assert bench.compare_rows(w, got, ref, rows)["outside_tolerance"] == 2


def test_cpulist_parsing():
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("") == set()


def test_numa_lookup_never_raises():
    # Without a GPU (or without the sysfs entries) the lookup reports why and
    # returns no CPU set; the e2e step then pins its buffers from where it runs.
    cpus, note = bench.gpu_numa_cpus(0)
    assert cpus is None or (isinstance(cpus, set) and cpus)
    assert isinstance(note, dict) and note


def test_dram_rate_from_recorded_traffic():
    r = bench.dram_rate(4281244331, 603.92, 6787.6)
    assert abs(r["dram_gbs"] - 4281244331 / 603.92e-6 / 1e9) < 0.01
    assert abs(r["dram_frac"] - r["dram_gbs"] / 6787.6) < 1e-4
    assert bench.dram_rate(None, 603.92, 6787.6) == {}
