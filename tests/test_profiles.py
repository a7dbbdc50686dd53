"""The committed profiler records are well formed (no GPU needed).

profiles/dram_traffic.json carries the DRAM bytes per launch that bench.py reports
as roofline traffic. Each record must add up, name a summary that exists and quotes
the same source hash, and state the algorithmic bytes of its workload.
"""
import json
import os

import synth
from memory_bound_row_rows_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORDS = os.path.join(ROOT, "profiles", "dram_traffic.json")


def algorithmic_bytes(key):
    """Algorithmic bytes per launch of the workload a record is keyed by."""
    if key.startswith("backward:"):
        w = synth.BACKWARD[key.split(":", 1)[1]]
        return 3 * w.M * w.N * synth.ELEM_BYTES[w.dtype]
    if key.startswith("rmsnorm:"):
        w = synth.RMSNORM[key.split(":", 1)[1]]
        return (3 * w.M * w.N + w.N) * synth.ELEM_BYTES[w.dtype]
    if key.startswith("split:"):  # the split plan's record of a softmax workload
        key = key.split(":", 1)[1]
    w = dict(synth.WORKLOADS, **synth.WIDE_FEW)[key]
    return 2 * w.M * w.N * w.elem_bytes


def test_records_are_consistent():
    with open(RECORDS) as f:
        records = json.load(f)
    keys = [k for k in records if not k.startswith("_")]
    assert keys
    for key in keys:
        r = records[key]
        assert r["plan"] in _build.PLAN_SOURCES, key
        assert r["dram_bytes_per_launch"] == r["dram_read"] + r["dram_write"], key
        assert r["algorithmic_bytes"] == algorithmic_bytes(key), key
        # Every input byte is read from DRAM about once (two of the three
        # matrices of a row-pair operation are inputs, one of the two of the
        # softmax): far above would be a re-read, below the capture is wrong.
        # Streamed kernels read their slices twice by design, the second time
        # mostly from L2: at most twice from DRAM.
        pair = key.startswith(("backward:", "rmsnorm:"))
        inputs = r["algorithmic_bytes"] * (2 / 3 if pair else 1 / 2)
        top = 2.0 if "stream" in r["kernel"] else 1.10
        assert 0.95 <= r["dram_read"] / inputs <= top, key
        summary = os.path.join(ROOT, r["summary"])
        assert os.path.exists(summary), key
        with open(summary) as f:
            assert r["source_hash"] in f.read(), "%s: summary quotes another hash" % key


def test_every_benchmark_workload_has_a_record():
    with open(RECORDS) as f:
        records = json.load(f)
    for name in synth.WORKLOADS:
        assert name in records, name
