"""bench.py on the CPU: its launch and kernel bookkeeping (read from the library's gdn_plan) for the named
workloads, and the reference arm's JSON line, run on the smallest workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_recurrence_delta_gb300 import inputs as I  # noqa: E402


@pytest.mark.parametrize("name,kernel,fwd,bwd", [
    ("delta_bf16_8x16x4096x64", "fwd_tc_kernel<delta>", 1, 4),    # chunked backward: prep, chain, grads, dA_log
    ("gated_bf16_8x16x4096x56_bwd", "fwd_tc_kernel<gated>", 1, 4),
    # forward: the time split by walks; backward: the chain in 4 segments (first walks, scan, second walks)
    ("delta_bf16_1x16x32768x64_bwd", "fwd_tc_kernel<delta>", 5, 6),
    ("delta_bf16_8x40x4096x32", "serial_fwd_kernel<bf16, delta>", 1, 4),       # narrow heads, 320 units
    ("delta_bf16_8x16x4096x128", "serial_fwd_kernel<bf16, delta>", 1, 6),      # 4 slabs: + sums of db, dc, dg, dbeta
    ("delta_bf16_decode_512x16x1x64", "decode_kernel", 1, 4),
])
def test_launch_bookkeeping(name, kernel, fwd, bwd):
    w = I.WORKLOADS[name]
    assert bench.fwd_kernel_name(w).startswith(kernel)
    assert bench.fwd_launches(w) == fwd
    assert bench.bwd_launches(w) == bwd


def test_split_chain_launches_from_residuals():
    """From the forward's residuals the split chain runs only its reverse sweep, in more segments, with the same
    kernels: prep, first walks, scan, second walks, gradients, dA_log sum."""
    w = I.WORKLOADS["delta_bf16_1x16x32768x64_bwd"]
    assert bench.plan(w, True).segments == 4 and bench.plan(w, 2).segments == 9
    assert bench.bwd_launches(w, saved=True) == 6
    assert bench.fwd_launches(w, saving=True) == 6   # the saving forward adds the residuals' fix-up
    assert bench.bwd_launches(I.WORKLOADS["delta_bf16_8x16x4096x64"], saved=True) == 4


def test_split_backward_launches_follow_the_runs():
    """The split (token-serial) backward sums G_p over runs of 512 tokens: one run per 512-token segment needs no
    partial sum."""
    w = I.custom(name="two_seg", mode="delta", dtype="bf16", B=1, H=64, T=1024, dk=64, dv=64, backward=True,
                 gate_logits=True)
    assert bench.tsplit_factor(w, True) == 2
    assert bench.bwd_launches(w) == 4 + 1 + 1 + 2        # states, G_p, reverse scan, backward + dA_log sum


def test_reference_arm_line():
    """--impl reference times the fp64 oracle on the host and prints one JSON line with the contract's keys."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "gated_f32_1x2x128x16", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["config"]["workload"] == "gated_f32_1x2x128x16"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["warmup"] >= 3 and line["steps"] == 3
