"""Writes csrc/fp4q_pairtab.cuh: per-block multiplier pairs for bf16 input.

The quantizer's codes are t = x' / s rounded to E2M1 (round to nearest even,
saturating at 6), with x' = u / S and both quotients rounded to binary32
("NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4 training",
"Technical design", scale levels 2 and 3; "Block-Scaled FP8 and FP4 Weight
Quantization", section 3).  When u and the outer amax A are bf16 values, S =
RN(A / (scale_max * 6)) has one of 128 significands sigma_m (m: the 7
mantissa bits of A; scale_max * 6 = 21 * 2^k), and s, an E4M3 or UE5M3
value, one of 8 significands sd_j = 1 + j / 8.  For every pair (j, m) this
script finds binary32 multipliers c1, c2 (a few ulps from 1 / sigma_m and
1 / sd_j) such that

    E2M1(RN(RN(u * c1) * c2)) == E2M1(RN(RN(u / sigma_m) / sd_j))

for EVERY bf16 u, by enumeration: only u with t in [0.2, 8] can differ (below
0.2 both give the code of 0, above 8 both saturate), and at exponent 0 for
sigma and sd that is every bf16 significand in a few binades.  Scaling u, S
and s by powers of two scales both sides alike while the intermediate stays
normal, which it does whenever t >= 0.2 (|x'| >= 0.2 * 2^-17).  So two
multiplies per value give the same codes as the two correctly rounded
divisions.  The arithmetic below is numpy binary32 (IEEE round to nearest
even, no contraction, subnormals kept).

Two more rows complete the table the kernels keep in shared memory: row 8
(c1 = 1, c2 = 0) for a zero inner scale, and row 9, the split reciprocal
(zh, zl) of sigma_m, zh = RD(1 / sigma), zl = RN(1 / sigma - zh), with which
the known-divisor method RN(u zh + RN(u zl)) gives RN(u / sigma) for bf16 u
(the block maxima); for sigma = 1 (zl = 0) row 9 holds zl = 2^-37 zh, which
changes no quotient that is normal (it stays below half an ulp).

The kernels copy a ready-made shared-memory image per scale format (kCtlTab,
one bulk copy): the ten rows with the exponent of S folded in (entry m of a
row gets ((127 + K - c) << 23) + (m << 16) added to c1, and to zh and zl:
S = sigma_m 2^(e_A - K + c) with c = 1 for m >= 40, K = 12 for E4M3 and 20
for UE5M3 scales; subtracting the bits of a bf16 amax A then gives the
multiplier for that S), the scale-code table (code -> row << 10 and the
negated exponent of s << 23), and the table of the form without an outer
scale (code -> c1, c2 / s of sigma = 1).

The table is a build input, committed beside the sources; run this script
to regenerate it (`python -m block_scaled_fp4_quantize_gb300.gen_pairtab`).
tests/test_pairtab.py checks the committed table the same way.
"""
import os
import sys
from fractions import Fraction

import numpy as np

F32 = np.float32
RANGE = 16  # ulps searched around 1 / sigma and 1 / sd


def sigma(m):
    """Significand in [1, 2) of RN((128 + m) / 21) (binary32 division)."""
    q = F32(128 + m) / F32(21)
    return F32(q * F32(0.25)) if q < 8 else F32(q * F32(0.125))


def inner_sig(j):
    return F32(1 + j / 8)


def e2m1_code(t):
    """Magnitude code of RNE-to-E2M1 with saturation (ties go to the even code)."""
    t = np.abs(t)
    return ((t > 0.25).astype(np.int8) + (t >= 0.75) + (t > 1.25) + (t >= 1.75) + (t > 2.5) + (t >= 3.5) + (t > 5.0))


def bf16_in(lo, hi):
    """Every positive bf16 value in [lo, hi] (as binary32)."""
    out = []
    for e in range(-8, 10):
        v = (np.arange(128, 256, dtype=np.float64) / 128.0) * 2.0 ** e
        out.append(v[(v >= lo) & (v <= hi)])
    return np.concatenate(out).astype(F32)


def cases(m, j):
    """(u, reference codes) of pair (j, m)."""
    sg, sd = sigma(m), inner_sig(j)
    u = bf16_in(0.2 * float(sg) * float(sd), 8.0 * float(sg) * float(sd))
    return u, e2m1_code((u / sg) / sd)


def exact(m, j, c1, c2):
    u, ref = cases(m, j)
    return bool((e2m1_code((u * F32(c1)) * F32(c2)) == ref).all())


def ulps(x, k):
    return (np.array([x], dtype=F32).view(np.int32) + np.int32(k)).view(F32)[0]


def search(m, j):
    sg, sd = sigma(m), inner_sig(j)
    b1, b2 = F32(1) / sg, F32(1) / sd
    u, ref = cases(m, j)
    d = np.arange(-RANGE, RANGE + 1)
    c1 = np.array([ulps(b1, k) for k in d], dtype=F32)
    c2 = np.array([ulps(b2, k) for k in d], dtype=F32)
    y = u[None, :] * c1[:, None]
    ok = (e2m1_code(y[:, None, :] * c2[None, :, None]) == ref[None, None, :]).all(axis=2)
    best = None
    for a in range(len(d)):
        for b in range(len(d)):
            if ok[a, b] and (best is None or abs(d[a]) + abs(d[b]) < abs(d[best[0]]) + abs(d[best[1]])):
                best = (a, b)
    if best is None:
        raise RuntimeError("no multiplier pair for j=%d m=%d" % (j, m))
    return c1[best[0]], c2[best[1]]


def bits(x):
    return int(np.array([x], dtype=F32).view(np.uint32)[0])


def round24(q, down):
    """q > 0 rounded to 24 significant bits, down or to nearest even."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    m = q * Fraction(2) ** (23 - e)
    n = m.numerator // m.denominator
    r = m - n
    if not down and (r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2)):
        n += 1
    return Fraction(n) * Fraction(2) ** (e - 23)


def rcp_split(m):
    """(zh, zl) bit patterns of the split reciprocal of sigma_m."""
    s = Fraction(sigma(m).item())
    zh = round24(1 / s, True)
    d = 1 / s - zh
    zl = round24(d, False) if d else zh / 2 ** 37
    return bits(F32(float(zh))), bits(F32(float(zl)))


def table():
    """[10][128] pairs as binary32 bit patterns: rows 0-7 (c1, c2), row 8
    (1, 0), row 9 (zh, zl)."""
    t = np.zeros((10, 128, 2), dtype=np.uint32)
    for j in range(8):
        for m in range(128):
            c1, c2 = search(m, j)
            t[j, m] = bits(c1), bits(c2)
    for m in range(128):
        t[8, m] = bits(F32(1)), 0
        t[9, m] = rcp_split(m)
    return t


def code_row(code, ue5m3):
    """(row, exponent) of an inner-scale code: s = (1 + row / 8) 2^e, row 8
    for s = 0."""
    ex, m3 = code >> 3, code & 7
    bias = 15 if ue5m3 else 7
    if ex:
        return m3, ex - bias
    if not m3:
        return 8, 0
    p = m3.bit_length() - 1  # subnormal s = m3 2^(-2 - bias)
    return (m3 << (3 - p)) & 7, p - 2 - bias


WORDS = 10 * 128 * 2 + 256 + 256 * 2  # per format: pair rows, code table, unit table


def ctl_image(t, ue5m3):
    """Shared-memory image of the whole-tile kernel for one scale format."""
    K = 20 if ue5m3 else 12
    w = []
    for row in range(10):
        for m in range(128):
            off = (((127 + K - (1 if m >= 40 else 0)) << 23) + (m << 16)) & 0xFFFFFFFF
            c1, c2 = int(t[row, m, 0]), int(t[row, m, 1])
            w += [(c1 + off) & 0xFFFFFFFF, ((c2 + off) & 0xFFFFFFFF) if row == 9 else c2]
    for code in range(256):
        row, e = code_row(code, ue5m3)
        w.append(((row << 10) | ((-e) << 23)) & 0xFFFFFFFF)
    for code in range(256):
        row, e = code_row(code, ue5m3)
        c1, c2 = int(t[row, 40, 0]), int(t[row, 40, 1])
        w += [c1, 0 if row == 8 else (c2 + ((-e) << 23)) & 0xFFFFFFFF]
    assert len(w) == WORDS
    return w


HEADER = """// fp4q_pairtab.cuh -- written by gen_pairtab.py; do not edit.
//
// kPairTab[j][m] = {c1, c2} (binary32 bits) for inner-scale significand
// 1 + j / 8 and outer-scale significand sigma_m = RN((128 + m) / 21) scaled
// into [1, 2): for every bf16 u the E2M1 code of RN(RN(u * c1) * c2) equals
// that of RN(RN(u / sigma_m) / (1 + j / 8)) (enumerated by the generator and
// by tests/test_pairtab.py).  Row 8: {1, 0} (a zero inner scale).  Row 9:
// {zh, zl}, the split reciprocal of sigma_m (zl = 2^-37 zh for sigma = 1).
//
// kCtlTab[f] (f = 0: E4M3 scales, 1: UE5M3) is the shared-memory image of the
// whole-tile kernel: the ten rows with the exponent of S folded in (entry m
// gets ((127 + K - c) << 23) + (m << 16) added to c1, and to zh and zl; c = 1
// for m >= 40, K = 12 / 20), then 256 words code -> (row << 10) | ((-e_s) <<
// 23), then 256 pairs code -> (c1, c2 / s) of sigma = 1.
#pragma once
#include <cstdint>

namespace fp4q {

__device__ const uint32_t __align__(16) kPairTab[10][128][2] = {
"""

CTL_WORDS = "constexpr int kCtlTabWords = %d;\n\n" % WORDS


def write(path):
    t = table()
    lines = [HEADER]
    for j in range(10):
        lines.append("    {  // %s\n" % ("j = %d" % j if j < 8 else ("zero inner scale" if j == 8 else "split reciprocal of sigma")))
        for m0 in range(0, 128, 4):
            lines.append("        " + " ".join("{0x%08Xu, 0x%08Xu}," % (t[j, m, 0], t[j, m, 1]) for m in range(m0, m0 + 4)) + "\n")
        lines.append("    },\n")
    lines.append("};\n\n")
    lines.append(CTL_WORDS)
    lines.append("__device__ const uint32_t __align__(16) kCtlTab[2][kCtlTabWords] = {\n")
    for f in range(2):
        img = ctl_image(t, f == 1)
        lines.append("    {  // %s scales\n" % ("UE5M3" if f else "E4M3"))
        for i in range(0, len(img), 8):
            lines.append("        " + " ".join("0x%08Xu," % v for v in img[i:i + 8]) + "\n")
        lines.append("    },\n")
    lines.append("};\n\n}  // namespace fp4q\n")
    with open(path, "w") as f:
        f.write("".join(lines))


if __name__ == "__main__":
    out = sys.argv[1] if len(sys.argv) > 1 else os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc",
                                                             "fp4q_pairtab.cuh")
    write(out)
    print(out)
