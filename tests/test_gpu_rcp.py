"""The cast-transpose kernel takes RN(1 / S) from the hardware reciprocal
approximation and one Markstein correction (rcp_markstein) instead of
rcp.rn.f32.  This test builds a small CUDA program that compares the two for
every binary32 of the range the kernel uses (2^-125 .. 2^125, both signs)
and requires no mismatch."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gpu_rcp_check.cu")
CSRC = os.path.join(ROOT, "block_scaled_fp4_quantize_gb300", "csrc")


@pytest.mark.gpu
def test_rcp_markstein_matches_ieee_reciprocal(tmp_path):
    exe = str(tmp_path / "gpu_rcp_check")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-I", CSRC, SRC, "-o", exe],
                   check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    m = re.search(r"checked (\d+) mismatches (\d+)", out.stdout)
    assert m, out.stdout
    assert int(m.group(1)) == 2 * (0x7E000000 - 0x01000000 + 1)
    assert int(m.group(2)) == 0, out.stdout
