"""The fast quantizer kernel replaces div.rn with two published exact
division methods.  These host tests check (1) that the reciprocal constants
in the kernel source are exactly RD(1/d) and RN(1/d - RD(1/d)), computed here
with rational arithmetic, and (2) that both methods reproduce the IEEE
correctly rounded quotient on sampled dividends across binades and signs,
using the same binary32 fma / mul on the host."""
import os
import re
import struct
import subprocess
from fractions import Fraction

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "block_scaled_fp4_quantize_gb300", "csrc", "fp4q_block.cuh")
CHECK = os.path.join(os.path.dirname(os.path.abspath(__file__)), "division_methods_check.c")


def _f(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def _b(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


def _rd(x):
    f = float(x)
    f = _f(_b(struct.unpack("<f", struct.pack("<f", f))[0]))
    while Fraction(f) > x:
        f = _f(_b(f) - 1)
    while Fraction(_f(_b(f) + 1)) <= x:
        f = _f(_b(f) + 1)
    return f


def _rn(x):
    if x == 0:
        return 0.0
    f = struct.unpack("<f", struct.pack("<f", float(x)))[0]
    c = [_f(_b(f) + d) for d in (-1, 0, 1)]
    return min(c, key=lambda v: (abs(Fraction(v) - x), _b(v) & 1))


def _split(d):
    hi = _rd(Fraction(1, d))
    return _b(hi), _b(_rn(Fraction(1, d) - Fraction(hi)))


def _kernel_constants():
    src = open(KERNEL).read()
    arr = {}
    for name in ("kRcpHi", "kRcpLo"):
        body = re.search(name + r"\[16\]\s*=\s*\{([^}]*)\}", src).group(1)
        arr[name] = [int(v.strip().rstrip("u"), 16) for v in body.split(",")]
    scal = {n: int(v, 16) for n, v in re.findall(r"(k\w+) = (0x[0-9A-Fa-f]+)u", src)}
    return arr, scal


def test_reciprocal_tables_are_exact():
    arr, scal = _kernel_constants()
    for M in range(1, 16):
        assert (arr["kRcpHi"][M], arr["kRcpLo"][M]) == _split(M), M
    assert (scal["kSixHi"], scal["kSixLo"]) == _split(6)
    assert (scal["kDenHiE4"], scal["kDenLoE4"]) == _split(2688)       # 448 * 6
    assert (scal["kDenHiU5"], scal["kDenLoU5"]) == _split(688128)     # 114688 * 6


def test_bmr_and_markstein_match_ieee_division(tmp_path):
    arr, _ = _kernel_constants()
    exe = str(tmp_path / "check")
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, CHECK, "-lm"],
                   check=True)
    args = []
    for M in range(1, 16):
        args += ["%08x" % arr["kRcpHi"][M], "%08x" % arr["kRcpLo"][M]]
    args += ["%08x" % v for v in _split(21)]
    r = subprocess.run([exe, "61"] + args, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bmr 0 of" in r.stdout and "markstein 0 of" in r.stdout
