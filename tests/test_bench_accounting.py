"""The benchmark's byte accounting and its ncu-traffic lookup (no GPU).

Algorithmic bytes of one GEMV are the packed codes (K/2 per row), the bf16
scales (2 per row and group) and the bf16 activations (2 per token and k);
the values below are that sum worked out for the five workloads."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_of_the_workloads():
    assert bench.algo_bytes(1, 256, 512, 128) == 65536 + 2048 + 1024 == 68608
    assert bench.algo_bytes(1, 4096, 4096, 128) == 8388608 + 262144 + 8192 == 8658944
    assert bench.algo_bytes(1, 14336, 4096, 128) == 29360128 + 917504 + 8192 == 30285824
    assert bench.algo_bytes(16, 14336, 4096, 128) == 29360128 + 917504 + 131072
    assert bench.algo_bytes(1, 4096, 14336, 128) == 29360128 + 917504 + 28672
    assert bench.algo_bytes(1, 163840, 4096, 128) == 335544320 + 10485760 + 8192 == 346038272


def test_int3_algorithmic_bytes_of_the_expert_matrices():
    # INT3: three bits per weight (3K/8 bytes per row), same scales and activations;
    # one MoE gate/up expert matrix is 1024 x 2304, the down matrix 2304 x 1024
    assert bench.algo_bytes3(0, 1024, 2304, 128) == 884736 + 36864
    assert bench.algo_bytes3(0, 2304, 1024, 128) == 884736 + 36864
    assert bench.algo_bytes3(1, 1024, 2304, 128) - bench.algo_bytes3(0, 1024, 2304, 128) == 4608


def test_all_bytes_add_zero_points_and_outputs():
    # zero points (1 byte per row and group) and the bf16 output
    assert bench.all_bytes(1, 4096, 4096, 128) - bench.algo_bytes(1, 4096, 4096, 128) == 131072 + 8192


def test_profiled_traffic_follows_the_kernel_source(monkeypatch):
    t = bench.profiled_traffic()
    text = open(bench.PROFILE_SUMMARY).read()
    if "kernel_source_sha256_16: %s" % bench.kernel_source_hash() in text:
        # captured on this source: DRAM traffic of a launch, at least its algorithmic bytes
        assert t is not None and t >= bench.algo_bytes(1, 4096, 4096, 128)
    else:
        assert t is None
    # a different kernel source: the stored counter no longer applies
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic() is None


def test_expert_gemv_bytes_count_each_distinct_expert_once():
    import numpy as np
    ids = np.array([[3, 7, 3, 9], [7, 7, 1, 3]], np.int32)   # experts 1, 3, 7, 9
    per4 = 1024 * 2304 // 2 + 1024 * (2304 // 128) * 2
    per3 = 1024 * 2304 * 3 // 8 + 1024 * (2304 // 128) * 2
    assert bench.moe_gemv_bytes(ids, 1024, 2304, 128, 4, False) == 4 * per4 + 2 * 2304 * 2
    assert bench.moe_gemv_bytes(ids, 1024, 2304, 128, 4, True) == 4 * per4 + 8 * 2304 * 2
    assert bench.moe_gemv_bytes(ids, 1024, 2304, 128, 3, False) == 4 * per3 + 2 * 2304 * 2
