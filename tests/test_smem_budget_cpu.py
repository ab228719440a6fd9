"""CPU: the forward kernel's shared-memory plan against the figures the page "FlashAttention
SM120 forward reuses the SM80 mainloop" prints (tests/golden/p1_smem_budget.txt): its
can_implement arithmetic for 128-row tiles and d = 128 in bf16 (Q + K + V with one K/V
stage, and with two), and the per-block limit of SM100-class GPUs, which GB300 shares.
The constants are read from the kernel header itself by a small host program
(tests/smem_budget_probe.cu), compiled here for sm_103a; nothing runs on a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KIB = 1024


def golden():
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", "p1_smem_budget.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, value = line.split()
                vals[key] = int(value)
    return vals


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc) and not shutil.which(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("probe") / "smem_budget_probe")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "exact_attention_forward_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "smem_budget_probe.cu"), "-o", exe],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    plan = {}
    for line in out.splitlines():
        name, *fields = line.split()
        plan[name] = {k: int(v) for k, v in (f.split("=") for f in fields)}
    return plan


def test_tile_arithmetic_reproduces_the_pages_budget(plan):
    g = golden()
    c = plan["bf16_d128"]  # 128 query rows x d = 128 bf16 per Q tile, 128 keys per K/V block
    assert c["tile_bytes"] == 128 * 128 * 2 and c["slot_bytes"] == 128 * 128 * 2
    assert c["tile_bytes"] + 2 * c["slot_bytes"] == g["q_k_v_one_stage"] * KIB
    assert c["tile_bytes"] + 2 * 2 * c["slot_bytes"] == g["q_k_v_two_kv_stages"] * KIB


def test_every_instance_fits_the_per_block_limit(plan):
    g = golden()
    for name, c in plan.items():
        # the byte count includes the barriers, item records and alignment slack
        assert c["smem_bytes"] <= g["per_block_limit_sm100"] * KIB, name
        # more than half the limit: one CTA, and one 512-column TMEM allocation, per SM
        assert 2 * c["smem_bytes"] > g["per_block_limit_sm100"] * KIB, name
        # the operand buffers alone: Q tiles, the K/V ring and the O staging tiles
        operands = c["tiles"] * (c["tile_bytes"] + c["stage_bytes"]) + c["stages"] * c["slot_bytes"]
        assert operands <= c["smem_bytes"], name


def test_the_bf16_plan_needs_the_sm100_class_budget(plan):
    # two Q tiles, four K/V stages and two O staging tiles: 224 KiB of operands, more than
    # any per-block limit of the SM80 or SM120 tables, within the SM100-class one
    g = golden()
    c = plan["bf16_d128"]
    operands = c["tiles"] * (c["tile_bytes"] + c["stage_bytes"]) + c["stages"] * c["slot_bytes"]
    assert operands == 224 * KIB
    assert operands > max(g["per_block_limit_sm80"], g["per_block_limit_sm120"]) * KIB
