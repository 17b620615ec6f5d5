"""The algorithmic bytes and FLOPs behind bench.py's roofline fractions (no GPU).

The Switch top-1 workload (T=8192, d=1024, E=64, d_ff=4096, k=1, capacity 160)
routes 8168 rows over all 64 experts with the seeded inputs.  Its expert FFN then
reads every expert's W1|W3 and W2 once (64 x 3 x 1024 x 4096 bf16), reads the
8168 gathered rows, writes H (8168 x 4096) and reads it back, and writes Y.  The
ncu record of that launch (profiles/) measures 1.779 GB of DRAM traffic against
these 1.778 GB.
"""
import numpy as np
import pytest

import bench
from workloads import WORKLOADS


def _switch_model(dtype="bf16"):
    wl = WORKLOADS["switch_top1_cap1.25"].with_(dtype=dtype)
    off = np.zeros(wl.E + 1, np.int64)
    off[-1] = 8168
    return bench.work_model(wl, off, 64)


def test_switch_ffn_bytes_and_flops():
    m, A, touched = _switch_model()
    weights = 64 * 3 * 1024 * 4096 * 2          # 1.611 GB
    x_perm = 8168 * 1024 * 2
    h_round_trip = 2 * 8168 * 4096 * 2
    y = 8168 * 1024 * 2
    assert (A, touched) == (8168, 64)
    assert m["ffn"]["bytes"] == weights + x_perm + h_round_trip + y == 1_777_893_376
    assert m["ffn"]["flops"] == 6 * 8168 * 1024 * 4096 == 205_554_450_432


def test_switch_layer_roofline():
    m, _, _ = _switch_model()
    layer_bytes = sum(m[s]["bytes"] for s in bench.STAGES)
    assert layer_bytes == 1_861_992_448
    # at the measured copy bandwidth the layer cannot take less than 0.286 ms
    assert layer_bytes / 6508.2e9 * 1e3 == pytest.approx(0.2861, abs=5e-5)


def test_fp8_weights_halve_the_weight_bytes():
    m16, _, _ = _switch_model("bf16")
    m8, _, _ = _switch_model("fp8w")
    weights16 = 64 * 3 * 1024 * 4096 * 2
    weights8 = 64 * (3 * 1024 * 4096 + 4 * (2 * 4096 + 1024))   # E4M3 codes + one fp32 scale per output channel
    assert m16["ffn"]["bytes"] - m8["ffn"]["bytes"] == weights16 - weights8


def test_fp8_up_projection_weight_bytes():
    # E4M3 W1|W3 with one fp32 scale per hidden column of each, bf16 W2
    m16, _, _ = _switch_model("bf16")
    m8, _, _ = _switch_model("fp8up")
    up16, up8 = 64 * 2 * 1024 * 4096 * 2, 64 * (2 * 1024 * 4096 + 4 * 2 * 4096)
    rows16 = 2 * 8168 * 1024 * 2                           # x_perm read, Y written (bf16)
    rows8 = 8168 * 1024 * (2 + 1 + 1) + 8168 * 1024 * 2    # quantised (read, write codes, read codes), Y
    assert m16["ffn"]["bytes"] - m8["ffn"]["bytes"] == (up16 - up8) + (rows16 - rows8)
    # the up projection's FLOPs count half at the FP8 rate
    assert m8["ffn"]["flops_bf16_equiv"] == 4 * 8168 * 1024 * 4096
