"""The tensor pipe's cost of an mbarrier wait between groups of tcgen05
MMAs, by how the issuing loop runs (tests/probes/mma_wait_cost.cu).

The attention kernels issue their MMAs from a whole warp, one elected lane
issuing, because with the loop in a lane-0 branch every wait between MMA
groups left the tensor pipe idle for about 150 cycles.  This test builds the
probe with nvcc, runs it, prints the cycles per step of each form and checks
the property the kernels rely on: waits in the warp-wide loop cost the pipe
almost nothing (within 5 % of the loop with no waits).
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_waits_in_a_warp_wide_issuing_loop_cost_the_tensor_pipe_almost_nothing():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "mma_wait_cost")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(ROOT, "attention_forward_online_gb300", "csrc"),
                        "-o", exe, os.path.join(ROOT, "tests", "probes", "mma_wait_cost.cu"),
                        "-lcuda"], check=True, capture_output=True, timeout=300)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(out.stdout)
    assert out.returncode == 0, out.stdout + out.stderr
    cyc = {int(m.group(1)): float(m.group(2))
           for m in re.finditer(r"mode (\d) err=0 bad=0 cycles_per_step (\d+)", out.stdout)}
    assert set(cyc) == {0, 1, 2}, out.stdout
    # 4 groups of 8 MMAs of 64 cycles each: 2048 cycles of tensor work a step
    assert 2000 < cyc[0] < 2300
    assert cyc[2] < 1.05 * cyc[0], cyc
    print(f"per wait: lane-0 loop {(cyc[1] - cyc[0]) / 4:.0f} cycles, "
          f"warp-wide loop {(cyc[2] - cyc[0]) / 4:.0f} cycles")
