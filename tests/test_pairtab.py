"""The per-block multiplier pairs of the bf16 fast path (csrc/fp4q_pairtab.cuh).

The kernels compute t = RN(RN(u * c1) * c2) in place of the two rounded
divisions t = RN(RN(u / S) / s) of the method ("NVFP4 / AMD-FP4 outer-block
(two-level) scaling for FP4 training", "Technical design": x' = u / S, then
the E2M1 code of x' / s).  This checks the committed table by enumeration:
for every pair (inner significand 1 + j / 8, outer significand sigma_m) and
every bf16 u whose t lies in [0.2, 8] (outside it both sides give the code of
0, or saturate), the E2M1 codes agree.  Reference quotients are IEEE binary32
divisions (numpy), the E2M1 rounding is pinned to the oracle's encoder.
"""
import os
import re
from fractions import Fraction

import numpy as np
import pytest
import oracle

F32 = np.float32
HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "block_scaled_fp4_quantize_gb300", "csrc",
                   "fp4q_pairtab.cuh")


def _hex_between(start, end):
    txt = open(HDR).read()
    body = txt[txt.index(start):txt.index(end) if end else len(txt)]
    return [int(v, 16) for v in re.findall(r"0x([0-9A-F]{8})u", body)]


def load_table():
    vals = _hex_between("kPairTab[10]", "kCtlTabWords")
    assert len(vals) == 10 * 128 * 2
    return np.array(vals, dtype=np.uint32).reshape(10, 128, 2)


def load_images():
    vals = _hex_between("kCtlTab[2]", None)
    assert len(vals) == 2 * 3328
    return np.array(vals, dtype=np.uint32).reshape(2, 3328)


def e2m1_mag(t):
    t = np.abs(t)
    return ((t > 0.25).astype(np.int8) + (t >= 0.75) + (t > 1.25) + (t >= 1.75) + (t > 2.5) + (t >= 3.5) + (t > 5.0))


def sigma(m):
    # S = RN(A / 2688) for A = (128 + m) * 2^4, i.e. RN((128 + m) / 168), scaled into [1, 2)
    s = F32(128 + m) / F32(168)
    while s < 1:
        s = F32(s * F32(2))
    return s


def bf16_in(lo, hi):
    out = []
    for e in range(-8, 10):
        v = (np.arange(128, 256, dtype=np.float64) / 128.0) * 2.0 ** e
        out.append(v[(v >= lo) & (v <= hi)])
    return np.concatenate(out).astype(F32)


def mismatches(tab, j, m):
    sg, sd = sigma(m), F32(1 + j / 8)
    c1, c2 = tab[j, m].view(F32)
    u = bf16_in(0.2 * float(sg) * float(sd), 8.0 * float(sg) * float(sd))
    ref = e2m1_mag((u / sg) / sd)
    fast = e2m1_mag((u * c1) * c2)
    return int((ref != fast).sum())


def test_e2m1_rounding_matches_the_oracle():
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    ts = []
    for x in ties + [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]:
        b = int(np.array([x], dtype=F32).view(np.uint32)[0])
        ts += [np.array([b + d], dtype=np.uint32).view(F32)[0] for d in (-2, -1, 0, 1, 2)]
    ts += list(np.random.default_rng(0).uniform(0, 8, 2000).astype(F32)) + [F32(0), F32(7.5), F32(1e30)]
    for t in ts:
        assert int(e2m1_mag(np.array([t], dtype=F32))[0]) == oracle.e2m1_rne(float(t)) & 7, t


def test_outer_significands_are_the_outer_scales_of_bf16_amax():
    # sigma_m is the significand of RN(A / (448 * 6)) for a bf16 A with mantissa m
    for m in range(128):
        A = F32((128 + m) / 128.0 * 2.0 ** 11)
        S = F32(A) / F32(2688)
        e = np.floor(np.log2(np.float64(S)))
        assert F32(S / F32(2.0 ** e)) == sigma(m)


def test_pair_table_is_exact_for_every_bf16_input():
    tab = load_table()
    bad = [(j, m, n) for j in range(8) for m in range(128) for n in [mismatches(tab, j, m)] if n]
    assert not bad, bad[:10]


def test_pair_table_check_has_teeth():
    # the enumeration catches a multiplier a few ulps off (planted in a copy)
    tab = load_table().copy()
    caught = 0
    for j, m in [(6, 58), (7, 68), (6, 100), (4, 47), (0, 10)]:
        for d in (-6, 6):
            t2 = tab.copy()
            t2[j, m, 0] = np.uint32(int(t2[j, m, 0]) + d)
            caught += mismatches(t2, j, m) > 0
    assert caught >= 5


def test_one_multiplier_is_not_enough():
    # for some pairs no single binary32 multiplier near 1 / (sigma sd) gives
    # the codes of the two rounded divisions: the second multiplier is needed
    for j, m in [(6, 58), (7, 68), (6, 100)]:
        sg, sd = sigma(m), F32(1 + j / 8)
        C = int(np.array([F32(1) / F32(np.float64(sg) * np.float64(sd))], dtype=F32).view(np.uint32)[0])
        u = bf16_in(0.2 * float(sg) * float(sd), 8.0 * float(sg) * float(sd))
        ref = e2m1_mag((u / sg) / sd)
        for d in range(-16, 17):
            c = np.array([C + d], dtype=np.uint32).view(F32)[0]
            assert (e2m1_mag(u * c) != ref).any(), (j, m, d)


def _r24(q, down=False):
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    m = q * Fraction(2) ** (23 - e)
    n = m.numerator // m.denominator
    if not down and (m - n > Fraction(1, 2) or (m - n == Fraction(1, 2) and n % 2)):
        n += 1
    return Fraction(n) * Fraction(2) ** (e - 23)


def test_rows_of_zero_scale_and_split_reciprocal():
    tab = load_table()
    assert (tab[8, :, 0] == 0x3F800000).all() and (tab[8, :, 1] == 0).all()
    for m in range(128):
        s = Fraction(float(sigma(m)))
        zh, zl = (Fraction(float(v)) for v in tab[9, m].view(F32))
        assert zh == _r24(1 / s, down=True)
        if zh * s == 1:   # sigma = 1: zl = 2^-37 zh stands in for 0
            assert m == 40 and zl == zh / 2 ** 37
            for k in range(128, 256):   # RN(u zh + RN(u zl)) = u for every bf16 significand
                u = Fraction(k, 128)
                assert _r24(u * zh + _r24(u * zl)) == _r24(u / s)
        else:
            assert zl == _r24(1 / s - zh)
            for k in range(128, 256):   # the known-divisor method: RN(u / sigma) for bf16 u
                u = Fraction(k, 128)
                assert _r24(u * zh + _r24(u * zl)) == _r24(u / s), (m, k)


def _f(b):
    return float(np.array([b & 0xFFFFFFFF], dtype=np.uint32).view(F32)[0])


def _b(x):
    return int(np.array([x], dtype=F32).view(np.uint32)[0])


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
def test_kernel_image_folds_the_outer_exponent(fmt):
    # c1 of the image less the bits of a bf16 amax A is c1 / 2^e_S, S = RN(A / (scale_max * 6))
    f = 1 if fmt == "ue5m3" else 0
    raw, img = load_table(), load_images()[f]
    rows = img[:2560].reshape(10, 128, 2)
    denom = F32(688128 if f else 2688)
    for m in range(0, 128, 3):
        for eA in (-80, -7, 0, 11, 40, 90):
            A = F32((128 + m) / 128.0 * 2.0 ** eA)
            S = F32(A) / denom
            eS = int(np.floor(np.log2(np.float64(S))))
            for row in (0, 3, 6, 7, 8, 9):
                got = _f(int(rows[row, m, 0]) - _b(A))
                assert got == _f(int(raw[row, m, 0])) * 2.0 ** -eS, (fmt, m, eA, row)
            zl = _f(int(rows[9, m, 1]) - _b(A))
            assert zl == _f(int(raw[9, m, 1])) * 2.0 ** -eS
            for row in range(9):
                assert rows[row, m, 1] == raw[row, m, 1]


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
def test_kernel_image_code_tables(fmt):
    f = 1 if fmt == "ue5m3" else 0
    raw, img = load_table(), load_images()[f]
    ctab, ntab = img[2560:2816], img[2816:].reshape(256, 2)
    for code in range(256):
        s = oracle.scale_decode(fmt, code)
        if not np.isfinite(s):
            continue
        w = int(ctab[code])
        row, e = (w & 0xFFFF) >> 10, -((w >> 23) - (512 if w >> 31 else 0))
        assert w & 0x7F03FF == 0
        if s == 0:
            assert row == 8 and ntab[code, 1] == 0
        else:
            assert row < 8 and s == (1 + row / 8) * 2.0 ** e, (fmt, code)
            assert _f(int(ntab[code, 1])) == _f(int(raw[row, 40, 1])) * 2.0 ** -e
        assert ntab[code, 0] == raw[row, 40, 0]
