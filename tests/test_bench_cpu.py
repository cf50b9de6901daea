"""bench.py's CPU-side bookkeeping: the oracle's work count for a whole
workload (the basis of cpu_baseline's extrapolated time) and the fields of
the cpu_baseline object, on the tiny workload."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_forward_02_gb300 import inputs  # noqa: E402


def _meta(name):
    q, k, v, meta = inputs.make_workload(name)
    meta["name"] = name
    return q, k, v, meta


def test_full_flops_equal_the_row_counts_summed_over_every_row():
    _, _, _, meta = _meta("tiny")
    B, H, N = meta["B"], meta["H"], meta["N"]
    every_row = np.stack([np.repeat(np.arange(B * H), N), np.tile(np.arange(N), B * H)], axis=1)
    for variants in ([False], [True], [False, True]):
        want = sum(bench.oracle_row_flops(meta, every_row, c) for c in variants)
        assert bench.oracle_full_flops(meta, variants) == want


def test_cpu_baseline_reports_rate_rows_and_extrapolated_time():
    q, k, v, meta = _meta("tiny")
    timer = bench.OracleTimer(q, k, v, meta, [False, True])
    cpu = bench.cpu_baseline_obj(timer, 0.2)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "TFLOP/s" and cpu["cores"] >= 1
    assert cpu["value"] > 0 and cpu["rows_per_s"] > 0
    # the extrapolation is the whole workload's oracle work at the measured rate
    full = bench.oracle_full_flops(meta, [False, True])
    assert abs(cpu["extrapolated_full_s"] - full / (cpu["value"] * 1e12)) <= 1e-9 * cpu["extrapolated_full_s"]
