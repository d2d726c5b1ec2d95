"""Host logic of bench.py, checked on the CPU.

The byte model is the roofline's numerator: the algorithmic bytes of a
verify launch are every packed target row (sum L + B rows, root and bonus
rows included) and, when sampling, every kept draft row (sum L), read once,
V logits each ("DFlash to DSpark in SGLang", "Ragged verify under full CUDA
graphs": the packed rows are the scheduled verify tokens plus one row per
request).  The mixed B=256 workload's figures are worked by hand here.
"""
import json

import numpy as np

import pytest
import torch

import bench
from confidence_driven_speculative_gb300 import workloads as W


def test_verify_bytes_of_the_mixed_workload():
    # B=256, gamma=16, V=129280 bf16, sum L = 768 (the cap): 1024 target rows
    # and 768 draft rows of 258,560 bytes, plus the small I/O
    B, g, V = 256, 16, 129280
    rows = (768 + 256) + 768
    small = 4 * (B * g + 5 * B + 2 * (B + 1) + 2 * B * (g + 1)) + 8 * 768
    assert bench.verify_bytes(B, 768, V, 2, True, g) == rows * V * 2 + small
    assert abs(bench.verify_bytes(B, 768, V, 2, True, g) / 1e6 - 463.4) < 0.1
    # greedy reads no draft rows
    assert bench.verify_bytes(B, 768, V, 2, False, g) == 1024 * V * 2 + small


def test_early_exit_bytes_counts_rows_up_to_the_first_rejection():
    a = torch.tensor([0, 2, 3], dtype=torch.int32)
    L = torch.tensor([3, 2, 5], dtype=torch.int32)
    V = 100
    # target rows 0..a_b: 1 + 3 + 4; draft rows min(a_b + 1, L_b): 1 + 2 + 4
    assert bench.early_exit_bytes(a, L, V, 2, True) == (8 + 7) * V * 2
    assert bench.early_exit_bytes(a, L, V, 2, False) == 8 * V * 2


def test_score_bytes_of_the_mixed_workload():
    # hidden [256, 16, 7168] bf16 = 58.7 MB read once, plus the head weight
    b = bench.score_bytes(256, 16, 7168, 2)
    assert b - 256 * 16 * 7168 * 2 == 4 * 7168 + 4 * (256 + 16) + 4 * (3 * 256 * 16 + 4 * 256)
    assert abs(b / 1e6 - 58.8) < 0.1


def test_whole_job_rate_is_units_over_the_slowest_rank():
    # K steps per rank, N ranks, the slowest rank's total time sets the rate
    assert bench.whole_job_rate(100, 4, 50.0) == pytest.approx(4 * 100 / 0.05)


def test_both_arms_name_the_workload_alike():
    cfg = bench.workload_config(W.MIXED_B256)
    assert cfg["workload"] == W.MIXED_B256.name
    assert (cfg["B"], cfg["gamma"], cfg["V"], cfg["d"]) == (256, 16, 129280, 7168)
    assert cfg["cap_T"] == 768 and cfg["cost_c"] == pytest.approx(0.35)


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The committed ncu traffic is reported only while the verify source
    it was taken on is unchanged; the figures are read from JSON."""
    good = tmp_path / "p.json"
    good.write_text(json.dumps({"traffic_bytes_per_launch": 123,
                                "source_sha256": bench.source_hash()}))
    monkeypatch.setattr(bench, "PROFILE_FILE", str(good))
    assert bench.profiled_traffic() == 123.0
    stale = tmp_path / "q.json"
    stale.write_text(json.dumps({"traffic_bytes_per_launch": 123,
                                 "source_sha256": "0000000000000000"}))
    monkeypatch.setattr(bench, "PROFILE_FILE", str(stale))
    assert bench.profiled_traffic() is None
    bad = tmp_path / "r.json"
    bad.write_text("traffic_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "PROFILE_FILE", str(bad))
    assert bench.profiled_traffic() is None
