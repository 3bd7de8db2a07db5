"""Exhaustive checks of device numerics that replace a general routine with
a shorter one, each a small CUDA program built here:

- rcp_markstein (RN(1 / S) from the hardware reciprocal approximation and
  one Markstein correction) against rcp.rn.f32 for every binary32 of the
  range the kernels use (2^-125 .. 2^125, both signs);
- enc_ue5m3 against the general scale encoder with the UE5M3 format for
  every finite binary32 v >= 0.

Each requires no mismatch."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(ROOT, "block_scaled_fp4_quantize_gb300", "csrc")


def _run_check(tmp_path, name):
    exe = str(tmp_path / name)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-I", CSRC,
                    os.path.join(HERE, name + ".cu"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    m = re.search(r"checked (\d+) mismatches (\d+)", out.stdout)
    assert m, out.stdout
    return int(m.group(1)), int(m.group(2)), out.stdout


@pytest.mark.gpu
def test_rcp_markstein_matches_ieee_reciprocal(tmp_path):
    n, bad, log = _run_check(tmp_path, "gpu_rcp_check")
    assert n == 2 * (0x7E000000 - 0x01000000 + 1)
    assert bad == 0, log


@pytest.mark.gpu
def test_enc_ue5m3_matches_general_encoder(tmp_path):
    n, bad, log = _run_check(tmp_path, "gpu_scale_check")
    assert n == 0x7F800000
    assert bad == 0, log


@pytest.mark.gpu
def test_hardware_encoders_match_the_oracle(tmp_path, orc):
    """The E2M1 (cvt.rn.satfinite.e2m1x2.f32) and E4M3 scale
    (cvt.rn.satfinite.e4m3x2.f32) conversions against the oracle's encoders
    for every finite binary32 >= 0, the stochastic E2M1 rounding against the
    oracle's for every binary32 in [0, 8] (one hashed random word each), the
    sign rule of both on the device, and Philox4x32-10 against the oracle's
    on 2^26 counters and keys."""
    so = orc.build()
    exe = str(tmp_path / "gpu_encoder_check")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", CSRC,
                    os.path.join(HERE, "gpu_encoder_check.cu"), "-o", exe, "-L", os.path.dirname(so), "-lorc",
                    "-Xlinker", "-rpath=" + os.path.dirname(so)], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    m = re.search(r"checked (\d+) mismatches (\d+)", out.stdout)
    assert m, out.stdout
    assert int(m.group(1)) == 2 * 0x7F800000 + 0x41000001 + (1 << 26)
    assert int(m.group(2)) == 0, out.stdout
