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


def _rn24(x):
    """x > 0 rounded to 24 significant bits, ties to even (exact rationals)."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    q = x / Fraction(2) ** (e - 23)
    n, r = divmod(q.numerator, q.denominator)
    r = Fraction(r, q.denominator)
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2):
        n += 1
    return n * Fraction(2) ** (e - 23)


def _rd24(x):
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    return (x // ulp) * ulp


def test_bmr_is_exact_for_outer_scales_of_bf16_amax():
    """The whole-tile cast-transpose kernel divides bf16 values u by an
    outer scale S = RN(A / (scale_max * 6)) whose amax A is itself a bf16
    value, so S's significand is that of RN(m / 21), m = 128 .. 255 (6 =
    3 * 2, 448 = 7 * 2^6, 114688 = 7 * 2^14).  For each of those 128
    divisors sigma, with zh = RD(1 / sigma) and zl = RN(1 / sigma - zh), the
    known-divisor method RN(u zh + RN(u zl)) must equal RN(u / sigma) for
    every dividend significand 1 .. 255 (exact rationals); and zl is at
    least 2^-30, so zl scaled by 2^-e stays normal for S < 2^90.  The
    device builds zh by a round-down division and zl as RN((1 - zh sigma) /
    sigma), with 1 - zh sigma exact: checked here too."""
    sigmas, zls = set(), []
    for m in range(128, 256):
        s = _rn24(Fraction(m, 21))
        while s >= 2:
            s /= 2
        sigmas.add(s)
        zh = _rd24(1 / s)
        d = 1 / s - zh
        zl = _rn24(d) if d else Fraction(0)
        if d:
            zls.append(zl)
            e = 1 - zh * s                                       # one fused multiply-add
            assert e == _rn24(e) and e / s == d
        for y in range(1, 256):
            got = _rn24(y * zh + (_rn24(y * zl) if zl else Fraction(0)))
            assert got == _rn24(Fraction(y) / s), (m, y)
    assert len(sigmas) == 128
    assert min(zls) >= Fraction(1, 2 ** 30)
