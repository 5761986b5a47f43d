"""The tensor-memory load with a min / max reduction the forward kernel
takes its row max from (tests/probes/tmem_ld_red.cu).

The kernel's unmasked score tiles get their row max (or min, for a negative
scale) from tcgen05.ld.red instead of a pass over the 128 scores; the
output stays bitwise that of the pass only if the reduction is exactly the
max / min of the values each thread receives.  This test builds the probe
with nvcc and runs it: every loaded value and every row's max and min must
match the stored tile bit for bit.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_tmem_load_reduction_is_the_exact_row_max_and_min():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "tmem_ld_red")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "-I", os.path.join(ROOT, "attention_forward_online_gb300", "csrc"),
                        "-o", exe, os.path.join(ROOT, "tests", "probes", "tmem_ld_red.cu")],
                       check=True, capture_output=True, timeout=300)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    print(out.stdout)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "values_mismatched 0 max_mismatched 0 min_mismatched 0" in out.stdout
