"""CPU: bench.py's roofline arithmetic for the tensor-bound workloads -- the FLOP and
exp2 counts and the two ceilings (tensor pipe, MUFU) reported beside the measurement."""
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_exp2_bound_of_the_causal_8k_pass():
    # B=2, H=32, S=8192, D=128, causal: 4 B H S^2 D / 2 FLOPs and one exp2 per visible
    # (query row, key) pair, B H S^2 / 2
    flops = 4.0 * 2 * 32 * 8192 * 8192 * 128 / 2
    r = bench.exp2_bound(flops, 128, 1928.9, 152, 2070.0, 32.0)
    assert math.isclose(r["exp2_per_launch"], 2 * 32 * 8192 * 8192 / 2)
    assert math.isclose(r["tensor_ms"], flops / 1928.9e12 * 1e3)
    assert math.isclose(r["exp2_ms"], 2 * 32 * 8192 * 8192 / 2 / (32 * 152 * 2070e6) * 1e3)
    assert r["limit"] == "tensor" and r["attainable_ms"] == r["tensor_ms"]
    assert 0.21 < r["exp2_ms"] < 0.22 and 0.56 < r["tensor_ms"] < 0.58


def test_exp2_bound_picks_the_larger_time():
    # head dim 8: 16x fewer FLOPs per exp2 than at 128, so the MUFU limits
    r = bench.exp2_bound(4.0 * 8 * 1e9, 8, 1928.9, 152, 2070.0, 32.0)
    assert r["limit"] == "exp2" and r["attainable_ms"] == r["exp2_ms"] > r["tensor_ms"]


def test_flop_count_of_the_workloads():
    from exact_attention_forward_gb300 import inputs
    w = inputs.WORKLOADS["bf16_causal_8k"]
    assert bench._flops(w, None) == 4.0 * 2 * 32 * 8192 * 8192 * 128 / 2
    w = inputs.WORKLOADS["bf16_noncausal_8k"]
    assert bench._flops(w, None) == 4.0 * 2 * 32 * 8192 * 8192 * 128


def test_per_sm_rates():
    r = bench._per_sm_rates(1000.0, [10, 20, 40, 0])
    assert r == {"median": 50.0, "min": 25.0, "max": 100.0}
