"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print (``tests/golden/page_values.json``), published known-answer
vectors, third-party format implementations (ml_dtypes, torch float8),
exact rational brute force, closed forms and invariants the pages state.
No test here touches a GPU.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_fp4_quantize_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
PAGE = json.load(open(os.path.join(GOLD, "page_values.json")))
GRID = [Fraction(v).limit_denominator(4) for v in PAGE["e2m1_grid"]["value"]]


def f32(v):
    return float(np.float32(v))


def bits_f32(b):
    return float(np.array([b], np.uint32).view(np.float32)[0])


def bf16_np(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32_np(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# E2M1
# ----------------------------------------------------------------------------

def test_e2m1_grid_is_the_printed_grid(orc):
    grid = PAGE["e2m1_grid"]["value"]
    for k in range(8):
        assert orc.e2m1_decode(k) == grid[k]
        assert orc.e2m1_decode(8 | k) == -grid[k]
        assert math.copysign(1.0, orc.e2m1_decode(8)) == -1.0


def _e2m1_nearest_fraction(t):
    """Exact nearest grid point by rational arithmetic, ties to the even code."""
    a = abs(Fraction(t))
    best = min(range(8), key=lambda k: (abs(a - GRID[k]), k % 2))
    return (8 if math.copysign(1.0, t) < 0 else 0) | best


def test_e2m1_rne_ties_and_saturation(orc):
    table = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for t, k in table.items():
        assert orc.e2m1_rne(t) == k
        assert orc.e2m1_rne(-t) == 8 | k
    for t in (6.0, 6.5, 7.0, 1e9, 3.0e38):
        assert orc.e2m1_rne(t) == 7
    assert orc.e2m1_rne(-0.1) == 8
    assert orc.e2m1_rne(-0.0) == 8
    assert orc.e2m1_rne(0.0) == 0


def _neighbourhood_f32(centres, ulps=64):
    out = []
    for c in centres:
        b = int(np.array([c], np.float32).view(np.uint32)[0])
        out.extend(range(max(0, b - ulps), b + ulps + 1))
    return np.array(out, np.uint32).view(np.float32)


def test_e2m1_rne_bruteforce_rational(orc):
    pts = [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0]
    vals = _neighbourhood_f32(pts, 8)
    rng = np.random.default_rng(0)
    vals = np.concatenate([vals, (rng.random(4000) * 8).astype(np.float32), -vals[::7]])
    for t in vals:
        assert orc.e2m1_rne(float(t)) == _e2m1_nearest_fraction(float(t)), t


def test_e2m1_rne_matches_ml_dtypes(orc):
    ml = pytest.importorskip("ml_dtypes")
    pts = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]
    vals = _neighbourhood_f32(pts, 256)
    rng = np.random.default_rng(1)
    vals = np.concatenate([vals, (rng.standard_normal(20000) * 3).astype(np.float32)])
    ref = vals.astype(ml.float4_e2m1fn).astype(np.float32)
    for t, r in zip(vals, ref):
        q = orc.e2m1_rne(float(t))
        assert orc.e2m1_decode(q & 7) == abs(float(r)), t
        assert (q >> 3) == int(np.signbit(t)), t


def test_e2m1_sr_endpoints_and_beyond(orc):
    for k, g in enumerate(PAGE["e2m1_grid"]["value"]):
        for w in (0, 1, 0x7FFFFFFF, 0xFFFFFFFF):
            assert orc.e2m1_sr(g, w) == k  # grid points never move
    for w in (0, 0xFFFFFFFF):
        assert orc.e2m1_sr(6.5, w) == 7
        assert orc.e2m1_sr(-100.0, w) == 15
    # 2.5 is half way between 2 and 3: up iff top 24 bits < 2^23
    assert orc.e2m1_sr(2.5, (0x7FFFFF << 8)) == 5
    assert orc.e2m1_sr(2.5, (0x800000 << 8)) == 4


# ----------------------------------------------------------------------------
# inner-scale formats
# ----------------------------------------------------------------------------

def test_e4m3_decode_matches_ml_dtypes_and_max(orc):
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(0x7F, dtype=np.uint8)
    ref = codes.view(ml.float8_e4m3fn).astype(np.float64)
    for c in codes:
        assert orc.scale_decode("e4m3", int(c)) == ref[c]
    assert orc.scale_decode("e4m3", 0x7E) == PAGE["e4m3_scale_max"]["value"]


def test_e4m3_encode_matches_ml_dtypes_and_torch(orc):
    ml = pytest.importorskip("ml_dtypes")
    vals_all = [orc.scale_decode("e4m3", c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals_all[:-1], vals_all[1:])]
    v = np.concatenate([_neighbourhood_f32([m for m in mids if m > 0], 3),
                        np.random.default_rng(2).random(20000).astype(np.float32) * 448,
                        np.exp2(np.random.default_rng(3).uniform(-14, 8.8, 20000)).astype(np.float32)])
    v = v[(v >= 0) & (v < 448)]
    ref_ml = v.astype(ml.float8_e4m3fn).view(np.uint8)
    ref_t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.scale_encode("e4m3", float(x)) for x in v], np.uint8)
    np.testing.assert_array_equal(got, ref_ml)
    np.testing.assert_array_equal(got, ref_t)
    for big in (448.0, 460.0, 1e6, 3e38):
        assert orc.scale_encode("e4m3", big) == 0x7E


def test_ue5m3_max_and_grid_structure(orc):
    vals = [orc.scale_decode("ue5m3", c) for c in range(0xFF)]
    assert vals[0xFE] == PAGE["ue5m3_scale_max"]["value"]
    assert all(b > a for a, b in zip(vals[:-1], vals[1:]))
    # each binade [2^e, 2^(e+1)) holds 8 values, 3 mantissa bits
    for c in range(0x08, 0xF8, 8):
        assert vals[c + 8] == 2 * vals[c]
        assert [vals[c + m] / vals[c] for m in range(8)] == [1 + m / 8 for m in range(8)]
    # subnormal step continues the smallest binade's spacing
    assert vals[1] == vals[9] - vals[8]


def test_ue5m3_is_e4m3_scaled_by_256(orc):
    """AMD-FP4 identity at the scale level: both grids have three mantissa
    bits and 114688 / 448 = 256, so on E4M3's normal range UE5M3 is E4M3
    shifted by 16 binades; encoding 256 v picks the same mantissa."""
    for c in range(0x08, 0x7F):
        assert orc.scale_decode("ue5m3", c + 128) == 256 * orc.scale_decode("e4m3", c)
    rng = np.random.default_rng(4)
    v = np.exp2(rng.uniform(-6, 8.8, 20000)).astype(np.float32)
    v = v[(v >= 2.0 ** -6) & (v < 448)]
    for x in v:
        assert orc.scale_encode("ue5m3", float(np.float32(x) * np.float32(256))) == \
            orc.scale_encode("e4m3", float(x)) + 128


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
def test_scale_encode_bruteforce_rational(orc, fmt):
    maxc = 0x7E if fmt == "e4m3" else 0xFE
    table = [Fraction(orc.scale_decode(fmt, c)) for c in range(maxc + 1)]
    rng = np.random.default_rng(5)
    lo, hi = (-12, 9) if fmt == "e4m3" else (-20, 17)
    v = np.exp2(rng.uniform(lo, hi, 3000)).astype(np.float32)
    mids = [(a + b) / 2 for a, b in zip(table[:-1], table[1:])]
    v = np.concatenate([v, _neighbourhood_f32([float(m) for m in mids[::5] if m > 0], 1)])
    for x in v:
        fx = Fraction(float(x))
        if fx >= table[-1]:
            want = maxc
        else:
            want = min(range(maxc + 1), key=lambda c: (abs(fx - table[c]), c % 2))
        assert orc.scale_encode(fmt, float(x)) == want, (fmt, x)


# ----------------------------------------------------------------------------
# Philox and the SR random stream
# ----------------------------------------------------------------------------

def test_philox_known_answers(orc):
    n = 0
    for line in open(os.path.join(GOLD, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = [int(v, 16) for v in line.split()]
        assert orc.philox4x32_10(f[0:4], f[4:6]) == f[6:10]
        n += 1
    assert n == 3


def test_sr_word_layout_and_uniformity(orc):
    # four consecutive elements share one Philox block
    out = orc.philox4x32_10([5, 0, 7, 1], [11, 0])
    assert [orc.sr_word(11, 7, 1, 20 + i) for i in range(4)] == out
    words = np.array([orc.sr_word(0, 3, 0, n) for n in range(1 << 16)], np.uint64)
    hist = np.bincount((words >> 24).astype(np.int64), minlength=256)
    exp = len(words) / 256
    chi2 = float(((hist - exp) ** 2 / exp).sum())
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)
    u = (words >> 8).astype(np.float64) / 2 ** 24
    assert abs(u.mean() - 0.5) < 6 * math.sqrt(1 / 12 / len(u))
    assert abs(u.var() - 1 / 12) < 0.003


# ----------------------------------------------------------------------------
# NVFP4 quantization: page-fixed statistics
# ----------------------------------------------------------------------------

def test_sr_mean_of_2p3(orc):
    """fp4-train 'Correctness': SR of 2.3 has mean 2.300; RTN gives 2.000."""
    pv = PAGE["sr_mean_of_2p3"]
    blk = np.full(16, 2.3, np.float32)
    blk[0] = 6.0  # block scale 6/6 = 1 exactly
    x = np.tile(blk, (62500, 2))
    kw = dict(G=1, M=62500, K=32, mode="none", fmt="e4m3")
    for rounding, want, tol in (("sr", pv["value"], pv["tol"]), ("rne", pv["rtn"], 0.0)):
        q = orc.quantize(x, rounding=rounding, seed=0, step=0)
        assert np.all(q["row_scales"] == 0x38)  # E4M3 1.0
        y = orc.dequantize(q["row_codes"], q["row_scales"], None, out_dtype="fp32", **kw)
        vals = y.reshape(62500, 2, 16)[:, :, 1:]
        assert abs(vals.mean() - want) <= tol, (rounding, vals.mean())
        assert set(np.unique(vals)) <= {2.0, 3.0}


def _ef_time_average(orc, x, steps):
    r = np.zeros((1, 1, 16), np.float32)
    total = 0.0
    for t in range(steps):
        q = orc.quantize(x, residual=r, mode="none", fmt="e4m3", rounding="rne")
        y = orc.dequantize(q["row_codes"], q["row_scales"], None, G=1, M=1, K=16, out_dtype="fp32")
        total += float(y.astype(np.float64).mean())
    return total / steps


def test_ef_time_average_of_2p3(orc):
    """fp4-train 'Correctness': RTN + error feedback time-averages to 2.297
    (= bf16(2.3) = 2.296875; in binary32 the same loop averages to 2.300)."""
    pv = PAGE["ef_time_average_of_2p3"]
    xb = np.full((1, 16), W.bf16_bits(2.296875), np.uint16)
    assert abs(_ef_time_average(orc, xb, 4000) - pv["value"]) <= pv["tol"]
    xf = np.full((1, 16), 2.3, np.float32)
    assert abs(_ef_time_average(orc, xf, 4000) - 2.3) <= pv["tol"]
    # without feedback RTN is stuck at one biased value
    q = orc.quantize(xb, mode="none", fmt="e4m3")
    y = orc.dequantize(q["row_codes"], q["row_scales"], None, G=1, M=1, K=16, out_dtype="fp32")
    assert np.all(y == 2.25)


def test_underflowing_block_quantizes_to_zero(orc):
    """fp4-train 'Requirements and limits': a block whose absmax is below the
    E4M3 scale range quantizes to zero."""
    x = np.full((1, 16), 2.0 ** -13, np.float32)  # a/6 < 2^-10, half the smallest E4M3
    x[0, 3] = -(2.0 ** -13)
    q = orc.quantize(x, mode="none", fmt="e4m3")
    assert q["row_scales"][0, 0, 0] == 0
    codes = np.concatenate([q["row_codes"] & 0xF, q["row_codes"] >> 4], axis=-1)
    assert set(np.unique(codes & 7)) == {0}
    y = orc.dequantize(q["row_codes"], q["row_scales"], None, G=1, M=1, K=16, out_dtype="fp32")
    assert np.all(y == 0)


def _unpack(codes):
    lo, hi = codes & 0xF, codes >> 4
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return out


@pytest.mark.parametrize("fmt,maxcode", [("e4m3", 0x7E), ("ue5m3", 0xFE)])
def test_outer_block_maps_amax_to_grid_top(orc, fmt, maxcode):
    """ALTO 'Technical design' item 1: the outer scale amax/(scale_max*6) puts
    the block's largest element at the top of both grids: its inner block gets
    the largest scale and the element itself codes to +-6."""
    x = bf16_np(W.lognormal((64, 256), 7, sigma=1.5))
    q = orc.quantize(x, mode="outer_block", ob=64, fmt=fmt, out_mask=3)
    xf = bf16_to_f32_np(x).reshape(64, 4, 64)
    codes = _unpack(q["row_codes"][0]).reshape(64, 4, 64)
    scales = q["row_scales"][0].reshape(64, 4, 4)
    A = np.abs(xf).max(axis=-1)
    S = q["row_outer"][0]
    np.testing.assert_array_equal(S, (A.astype(np.float32) / np.float32(6 * (448 if fmt == "e4m3" else 114688))))
    arg = np.abs(xf).argmax(axis=-1)
    for i in range(64):
        for j in range(4):
            assert scales[i, j, arg[i, j] // 16] == maxcode
            assert codes[i, j, arg[i, j]] & 7 == 7


def test_amdfp4_identity_on_well_ranged_data(orc):
    """ALTO 'Key properties': AMD-FP4 outer-block equals NVFP4 outer-block run
    on the UE5M3 grid; on well-ranged data the codes and dequantized values
    are identical, the outer scales differ by exactly 256."""
    x = bf16_np(W.moe_experts(G=2, M=128, K=192, experts=[3, 4]))
    kw = dict(mode="outer_block", ob=64, outer_2d=True, out_mask=3)
    a = orc.quantize(x, fmt="e4m3", **kw)
    b = orc.quantize(x, fmt="ue5m3", **kw)
    np.testing.assert_array_equal(a["tile_outer"], b["tile_outer"] * np.float32(256))
    well = a["row_scales"] >= 0x08  # E4M3-normal inner scales
    np.testing.assert_array_equal(a["row_codes"][np.repeat(well, 8, -1)],
                                  b["row_codes"][np.repeat(well, 8, -1)])
    np.testing.assert_array_equal(a["row_scales"][well].astype(int) + 128, b["row_scales"][well])
    dq = dict(G=2, M=128, K=192, mode="outer_block", ob=64, outer_2d=True, out_dtype="fp32")
    ya = orc.dequantize(a["row_codes"], a["row_scales"], {"tile_outer": a["tile_outer"]}, fmt="e4m3", **dq)
    yb = orc.dequantize(b["row_codes"], b["row_scales"], {"tile_outer": b["tile_outer"]}, fmt="ue5m3", **dq)
    wel = np.repeat(well, 16, -1)
    np.testing.assert_array_equal(ya[wel], yb[wel])
    assert well.mean() > 0.9


def test_amdfp4_divergence_only_where_e4m3_underflows(orc):
    """Same property on data whose dynamic range inside an outer block exceeds
    E4M3's: blocks may differ only where the E4M3 inner scale is subnormal."""
    rng = np.random.default_rng(9)
    xf = rng.standard_normal((64, 8, 16)).astype(np.float32)
    shrink = np.where(rng.random((64, 8, 1)) < 0.3, 10.0 ** -rng.uniform(3.5, 7, (64, 8, 1)), 1.0)
    x = bf16_np(torch.from_numpy((xf * shrink).astype(np.float32).reshape(64, 128)).to(torch.bfloat16))
    kw = dict(mode="outer_block", ob=64, out_mask=1)
    a = orc.quantize(x, fmt="e4m3", **kw)
    b = orc.quantize(x, fmt="ue5m3", **kw)
    differ = np.any((a["row_codes"] != b["row_codes"]).reshape(1, 64, 8, 8), axis=-1)
    sub = a["row_scales"] < 0x08
    assert differ.any()
    assert not np.any(differ & ~sub)


def test_tensorwise_is_one_outer_block(orc):
    """Tensorwise scaling is the outer-block machinery with a single block
    covering the tensor (ALTO 'Background')."""
    x = bf16_np(W.uniform_bf16((1, 256), 3))
    a = orc.quantize(x, mode="tensorwise", fmt="e4m3")
    b = orc.quantize(x, mode="outer_block", ob=256, fmt="e4m3")
    np.testing.assert_array_equal(a["row_codes"], b["row_codes"])
    np.testing.assert_array_equal(a["row_scales"], b["row_scales"])
    assert a["tile_outer"][0] == b["row_outer"].ravel()[0]


# ----------------------------------------------------------------------------
# invariants of the blog's layout discussion
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode,ob,outer_2d", [("none", 0, False), ("tensorwise", 0, False),
                                              ("outer_block", 32, True), ("outer_block", 64, True)])
def test_2d_scaling_is_transpose_consistent(orc, mode, ob, outer_2d):
    """Block-Scaled FP8 and FP4 Weight Quantization, section 6: with 16x16
    inner tiles (and 2-D or no outer scales) the columnwise buffers are the
    transposes of the rowwise ones."""
    x = bf16_np(W.moe_experts(G=1, M=128, K=192, experts=[1]))
    q = orc.quantize(x, mode=mode, ob=ob, outer_2d=outer_2d, inner_2d=True, out_mask=3)
    rc, cc = _unpack(q["row_codes"]), _unpack(q["col_codes"])
    np.testing.assert_array_equal(rc.transpose(0, 2, 1), cc)
    rs = np.repeat(q["row_scales"], 16, -1)
    cs = np.repeat(q["col_scales"], 16, -1)
    np.testing.assert_array_equal(rs.transpose(0, 2, 1), cs)


def test_1d_scaling_is_direction_dependent(orc):
    """Section 4 of the same page: 1-D blocks group different neighbours in
    the two directions, so the columnwise codes are not a transpose."""
    x = bf16_np(W.moe_experts(G=1, M=128, K=192, experts=[1]))
    q = orc.quantize(x, mode="outer_block", ob=64, outer_2d=True, out_mask=3)
    assert np.any(_unpack(q["row_codes"]).transpose(0, 2, 1) != _unpack(q["col_codes"]))


@pytest.mark.parametrize("mode,ob", [("none", 0), ("outer_block", 64), ("tensorwise", 0)])
def test_rowwise_1d_is_token_permutation_invariant(orc, mode, ob):
    """Section 7: per-token 1-D scaling commutes with a token permutation."""
    x = bf16_np(W.activations(M=128, K=192, n_cols=2, n_rows=1))
    perm = np.random.default_rng(6).permutation(128)
    a = orc.quantize(x, mode=mode, ob=ob)
    b = orc.quantize(np.ascontiguousarray(x[perm]), mode=mode, ob=ob)
    np.testing.assert_array_equal(a["row_codes"][0][perm], b["row_codes"][0])
    np.testing.assert_array_equal(a["row_scales"][0][perm], b["row_scales"][0])


def test_2d_tiles_break_permutation_invariance(orc):
    x = bf16_np(W.activations(M=128, K=192, n_cols=2, n_rows=1))
    perm = np.random.default_rng(6).permutation(128)
    kw = dict(mode="outer_block", ob=64, outer_2d=True)
    a = orc.quantize(x, **kw)
    b = orc.quantize(np.ascontiguousarray(x[perm]), **kw)
    assert np.any(a["row_codes"][0][perm] != b["row_codes"][0])


# ----------------------------------------------------------------------------
# internal consistency of the oracle's own entry points
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kw", [dict(mode="outer_block", ob=64, outer_2d=True, out_mask=3),
                                dict(mode="outer_block", ob=32, out_mask=3),
                                dict(mode="tensorwise", out_mask=3)])
def test_precomputed_outer_scale_is_equivalent(orc, kw):
    """ALTO 'Implementation': a returned outer scale, passed back as the
    precomputed scale, reproduces the quantization bit for bit."""
    x = bf16_np(W.activations(M=64, K=128, n_cols=1, n_rows=1))
    a = orc.quantize(x, **kw)
    pre = {k: a[k] for k in ("row_outer", "col_outer", "tile_outer")}
    b = orc.quantize(x, use_precomputed=True, precomputed=pre, **kw)
    for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
        np.testing.assert_array_equal(a[k], b[k])


def test_grid_values_round_trip_exactly(orc):
    """Values already on the E2M1 x E4M3 grid, with a +-6 in every block so
    the block scale is exact, survive quantize-dequantize unchanged."""
    rng = np.random.default_rng(8)
    grid = np.array(PAGE["e2m1_grid"]["value"], np.float32)
    e4 = np.array([orc.scale_decode("e4m3", c) for c in range(0x10, 0x7E)], np.float32)
    blocks = []
    for _ in range(256):
        s = rng.choice(e4)
        v = grid[rng.integers(0, 8, 16)] * np.where(rng.random(16) < 0.5, -1, 1).astype(np.float32)
        v[rng.integers(0, 16)] = 6.0 * (1 if rng.random() < 0.5 else -1)
        blocks.append(v * s)
    x = np.concatenate(blocks).astype(np.float32).reshape(16, 256)
    y, _ = orc.qdq(x, mode="none")
    np.testing.assert_array_equal(y[0], x)


@pytest.mark.parametrize("orient", [1, 2])
@pytest.mark.parametrize("kw", [dict(mode="none"), dict(mode="tensorwise"),
                                dict(mode="outer_block", ob=32),
                                dict(mode="outer_block", ob=64, outer_2d=True),
                                dict(mode="outer_block", ob=16, inner_2d=True)])
def test_qdq_equals_dequantize_of_quantize(orc, orient, kw):
    x = bf16_np(W.lognormal((64, 128), 11, sigma=1.0))
    q = orc.quantize(x, out_mask=orient, **kw)
    name = "row" if orient == 1 else "col"
    y1 = orc.dequantize(q[name + "_codes"], q[name + "_scales"], q, G=1, M=64, K=128, orient=orient,
                        out_dtype="bf16", mode=kw["mode"], ob=kw.get("ob", 0),
                        outer_2d=kw.get("outer_2d", False))
    y2, _ = orc.qdq(x, orient=orient, **kw)
    if orient == 2:
        y1 = y1.transpose(0, 2, 1)
    np.testing.assert_array_equal(y1, y2)


def test_rne_codes_minimise_error(orc):
    """Brute force on a small tensor: every RNE code is a nearest grid point of
    x'/s, and every inner scale is the nearest E4M3 value of amax/6."""
    x = bf16_np(W.uniform_bf16((8, 64), 12))
    q = orc.quantize(x, mode="none")
    xf = bf16_to_f32_np(x).reshape(8, 4, 16)
    codes = _unpack(q["row_codes"][0]).reshape(8, 4, 16)
    e4 = [Fraction(orc.scale_decode("e4m3", c)) for c in range(0x7F)]
    for i in range(8):
        for b in range(4):
            a = Fraction(float(np.float32(np.abs(xf[i, b]).max()) / np.float32(6)))
            sc = q["row_scales"][0, i, b]
            assert abs(e4[sc] - a) == min(abs(v - a) for v in e4)
            s = float(e4[sc])
            for j in range(16):
                t = Fraction(float(np.float32(xf[i, b, j]) / np.float32(s)))
                got = abs(GRID[codes[i, b, j] & 7] - abs(t))
                assert got == min(abs(g - abs(t)) for g in GRID)


def test_error_feedback_residual_is_the_rounding_error(orc):
    x = np.random.default_rng(13).standard_normal((4, 64)).astype(np.float32)
    r = np.zeros((1, 4, 64), np.float32)
    q = orc.quantize(x, residual=r, mode="outer_block", ob=32)
    y = orc.dequantize(q["row_codes"], q["row_scales"], q, G=1, M=4, K=64, out_dtype="fp32",
                       mode="outer_block", ob=32)
    np.testing.assert_array_equal(r, (x[None] - y).astype(np.float32))


def test_bf16_rounding_matches_torch(orc):
    v = np.random.default_rng(14).standard_normal(5000).astype(np.float32) * 1e3
    want = bf16_np(torch.from_numpy(v).to(torch.bfloat16))
    got = np.array([orc.f32_to_bf16(float(a)) for a in v], np.uint16)
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------------------
# MXFP4 fake-quantization
# ----------------------------------------------------------------------------

def _mx_reference_block(vals_bits):
    """Independent statement by exact rationals: the scale exponent is the
    least E with 6 * 2^E >= max(amax, 6*2^-126), capped at 125; each value is
    the nearest grid point of x / 2^E, ties to the even code."""
    vals = [bits_f32(int(b) << 16) for b in vals_bits]
    if any(not math.isfinite(v) for v in vals):
        return [0x7FC0] * len(vals)
    A = max(Fraction(abs(v)) for v in vals)
    Ac = max(A, Fraction(6) * Fraction(2) ** -126)
    E = -126
    while Fraction(6) * Fraction(2) ** E < Ac:
        E += 1
    E = min(E, 125)
    out = []
    for v in vals:
        q = _e2m1_nearest_fraction(float(Fraction(v) / Fraction(2) ** E)) if v != 0 else \
            (8 if math.copysign(1, v) < 0 else 0)
        mag = GRID[q & 7] * Fraction(2) ** E
        f = float(mag) * (-1 if q & 8 else 1)
        b = int(np.array([f], np.float32).view(np.uint32)[0])
        assert b & 0xFFFF == 0
        out.append(b >> 16)
    return out


def test_mxfp4_all_bf16_patterns(orc):
    x = bf16_np(W.all_bf16_patterns())
    y = orc.mxfp4_fake_quantize(x)[0]
    for r in range(256):
        for b in range(8):
            want = _mx_reference_block(x[r, 32 * b:32 * b + 32])
            assert list(y[r, 32 * b:32 * b + 32]) == want, (r, b)


def _mx_one(orc, vals):
    x = np.zeros((1, 32), np.uint16)
    x[0, :len(vals)] = vals
    return orc.mxfp4_fake_quantize(x)[0, 0]


def test_mxfp4_page_edge_values(orc):
    b = W.bf16_bits
    # the 2^-127 grid point survives; 2^-128 ties to zero; 2^-133 flushes
    assert _mx_one(orc, [0x0040])[0] == 0x0040
    assert _mx_one(orc, [0x0020])[0] == 0x0000
    assert _mx_one(orc, [0x8001])[0] == 0x8000
    # signed zeros keep their sign
    y = _mx_one(orc, [0x8000, 0x0000, b(1.0)])
    assert (y[0], y[1]) == (0x8000, 0x0000)
    # inf / NaN poison the whole block
    for bad in (0x7F80, 0xFF80, 0x7FC1):
        assert np.all(_mx_one(orc, [b(1.0), bad]) == 0x7FC0)
    # cap: amax = 6*2^125 is exact; one ulp more saturates at 6*2^125
    cap = b(6.0 * 2.0 ** 125)
    assert _mx_one(orc, [cap])[0] == cap
    assert _mx_one(orc, [cap + 1])[0] == cap
    assert orc.mxfp4_exponent(float(bits_f32((cap + 1) << 16))) == PAGE["mxfp4_scale_cap_exponent"]["value"]
    # floor: any amax at or below the 6*2^-126 clamp uses 2^-126
    assert orc.mxfp4_exponent(0.0) == PAGE["mxfp4_scale_floor_exponent"]["value"]
    assert orc.mxfp4_exponent(6.0 * 2.0 ** -126) == -126
    assert orc.mxfp4_exponent(6.0 * 2.0 ** -126 * (1 + 2 ** -7)) == -125


@pytest.mark.parametrize("k", [-100, -3, 0, 7, 90])
def test_mxfp4_threshold_triples(orc, k):
    at = W.bf16_bits(6.0 * 2.0 ** k)
    for top, want in ((at - 1, k), (at, k), (at + 1, k + 1)):
        assert orc.mxfp4_exponent(bits_f32(top << 16)) == want


def test_mxfp4_is_idempotent_and_exact_in_bf16(orc):
    x, _ = W.mxfp4_weight(M=64, K=4096, frac=0.05)
    xb = bf16_np(x)
    y1 = orc.mxfp4_fake_quantize(xb)[0]
    y2 = orc.mxfp4_fake_quantize(y1)[0]
    poisoned = np.any((xb.reshape(64, -1, 32) & 0x7F80) == 0x7F80, axis=-1)
    keep = ~np.repeat(poisoned, 32, -1)
    np.testing.assert_array_equal(y1[keep], y2[keep])
    y32 = orc.mxfp4_fake_quantize(xb, out_dtype="fp32")[0]
    f = bf16_to_f32_np(y1)
    np.testing.assert_array_equal(f[keep], y32[keep])  # bf16 output is exact


def test_columnwise_outer_scale_is_the_column_block_amax(orc):
    """Columnwise = the rowwise method applied to x transposed (blog section 4):
    the 1-D columnwise outer scale is the amax of an ob x 1 column segment."""
    x = bf16_np(W.lognormal((128, 64), 15, sigma=1.5))
    q = orc.quantize(x, mode="outer_block", ob=64, out_mask=2)
    xf = bf16_to_f32_np(x).astype(np.float32)
    A = np.abs(xf).reshape(2, 64, 64).max(axis=1)          # [M/ob, K]
    np.testing.assert_array_equal(q["col_outer"][0], (A.T / np.float32(2688)).astype(np.float32))
    xt = np.ascontiguousarray(x.T)
    r = orc.quantize(xt, mode="outer_block", ob=64, out_mask=1)
    np.testing.assert_array_equal(q["col_codes"][0], r["row_codes"][0])
    np.testing.assert_array_equal(q["col_scales"][0], r["row_scales"][0])


def _mx_reference_block_f32(vals):
    if any(not math.isfinite(v) for v in vals):
        return None
    A = max(Fraction(abs(float(v))) for v in vals)
    Ac = max(A, Fraction(6) * Fraction(2) ** -126)
    E = -126
    while Fraction(6) * Fraction(2) ** E < Ac:
        E += 1
    E = min(E, 125)
    out = []
    for v in vals:
        v = float(v)
        q = _e2m1_nearest_fraction(float(Fraction(v) / Fraction(2) ** E)) if v != 0 else \
            (8 if math.copysign(1, v) < 0 else 0)
        f = float(GRID[q & 7] * Fraction(2) ** E) * (-1 if q & 8 else 1)
        out.append(np.float32(f))
    return out


def test_mxfp4_fp32_input_bruteforce(orc):
    rng = np.random.default_rng(16)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-130, 120, (16, 1)))).astype(np.float32)
    x[3, 5] = np.float32(6.0 * 2.0 ** 125) * np.float32(1.25)
    y = orc.mxfp4_fake_quantize(x)[0]
    for r in range(16):
        for b in range(8):
            want = _mx_reference_block_f32(x[r, 32 * b:32 * b + 32])
            got = y[r, 32 * b:32 * b + 32]
            np.testing.assert_array_equal(got.view(np.uint32), np.array(want, np.float32).view(np.uint32))


# ----------------------------------------------------------------------------
# MXFP4 projection re-encoded as MXFP8 ([TEQAT] "Design"; MXFP8 per the OCP
# MX v1.0 reading stated in the oracle)
# ----------------------------------------------------------------------------

def _e4m3_decode_torch(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> float64 with torch's float8_e4m3fn (an independent decoder)."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _mxfp8_decode(codes, scales, axis_len):
    v = _e4m3_decode_torch(codes)
    X = scales.astype(np.int64) - 127
    return v * np.exp2(np.repeat(X, 32, axis=-1)).reshape(v.shape)


def _wide_range_bf16(shape, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(*shape, generator=g) * torch.exp2(torch.randint(-120, 120, (shape[0], 1), generator=g).float())
    return x.to(torch.bfloat16)


def test_mxfp8_rowwise_encoding_of_the_projection_is_lossless(orc):
    """[TEQAT] "Design": the MXFP8 rowwise encoding of the projected weight is
    bitwise lossless -- decoding codes and scales gives the projection back
    exactly (all bf16 patterns and a wide-range tensor; poisoned blocks aside)."""
    for x in (W.all_bf16_patterns(), _wide_range_bf16((64, 256), 21)):
        xb = x.view(torch.int16).numpy().view(np.uint16)
        out = orc.mxfp4_project_mxfp8(xb, out_dtype="fp32", out_mask=1)
        y = orc.mxfp4_fake_quantize(xb, out_dtype="fp32")[0]     # the separately pinned projection
        assert (out["y"][0].view(np.uint32) == y.view(np.uint32)).all()
        dec = _mxfp8_decode(out["row_codes"][0], out["row_scales"][0], 32)
        ok = np.isfinite(y)
        assert (dec[ok] == y[ok].astype(np.float64)).all()
        blocks = ~np.isfinite(y).reshape(y.shape[0], -1, 32).all(axis=2)
        assert (out["row_scales"][0][blocks] == 0xFF).all()
        assert (out["row_codes"][0].reshape(y.shape[0], -1, 32)[blocks] == 0x7F).all()


def test_mxfp8_exponent_rule(orc):
    """X = floor(log2 A) - 8, clamped to [-127, 127]; A = 0 gives -127."""
    rng = np.random.default_rng(5)
    vals = list(np.exp2(rng.uniform(-140, 130, 2000))) + [2.0 ** k for k in range(-140, 128)] + \
        [2.0 ** k * (2 - 2 ** -20) for k in range(-130, 127)]
    for A in vals:
        X = orc.mxfp8_exponent(float(A))
        f = Fraction(A)  # exact floor(log2 A) from the rational value
        fl = f.numerator.bit_length() - f.denominator.bit_length()
        if Fraction(2) ** fl > f:
            fl -= 1
        assert X == min(max(fl - 8, -127), 127), (A, X, fl)
    assert orc.mxfp8_exponent(0.0) == -127


def test_mxfp8_columnwise_elements_match_torch_float8(orc):
    """Columnwise blocks mix rows with different MXFP4 exponents: the element
    bytes are torch's float8_e4m3fn rounding of v / 2^X (never above 448 for
    projected values), and the re-quantization error is within half an E4M3
    step."""
    x = _wide_range_bf16((64, 128), 22)
    x[5, 7] = float("nan")
    xb = x.view(torch.int16).numpy().view(np.uint16)
    out = orc.mxfp4_project_mxfp8(xb, out_dtype="fp32", out_mask=2)
    y = out["y"][0].astype(np.float64)                     # [M, K]
    codes, scales = out["col_codes"][0], out["col_scales"][0]  # [K, M], [K, M/32]
    for k in range(128):
        for b in range(2):
            v = y[32 * b:32 * b + 32, k]
            if not np.isfinite(v).all():
                assert scales[k, b] == 0xFF and (codes[k, 32 * b:32 * b + 32] == 0x7F).all()
                continue
            X = int(scales[k, b]) - 127
            t = v * 2.0 ** -X
            assert np.abs(t).max() <= 448
            ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert (codes[k, 32 * b:32 * b + 32] == ref).all(), (k, b)
            dec = _e4m3_decode_torch(codes[k, 32 * b:32 * b + 32]) * 2.0 ** X
            assert (np.abs(dec - v) <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** (X - 10))).all()


def test_mxfp8_zero_and_signed_zero_blocks(orc):
    x = np.zeros((32, 64), np.uint16)
    x[:, 32:] = 0x8000                                       # -0 in the second block
    out = orc.mxfp4_project_mxfp8(x, out_dtype="bf16")
    assert (out["row_scales"][0] == 0).all()                # X = -127 for all-zero blocks
    assert (out["row_codes"][0][:, :32] == 0x00).all() and (out["row_codes"][0][:, 32:] == 0x80).all()
    assert (out["col_codes"][0][:32] == 0x00).all() and (out["col_codes"][0][32:] == 0x80).all()


# ----------------------------------------------------------------------------
# Random Hadamard transform along M before the columnwise quantization
# ([ALTO] "Op-level test coverage": outer-block x M-axis Hadamard; the
# transform itself is this build's reading, stated in the oracle)
# ----------------------------------------------------------------------------

def _sylvester16():
    H = np.ones((16, 16), dtype=object)
    for i in range(16):
        for k in range(16):
            H[i, k] = -1 if bin(i & k).count("1") % 2 else 1
    return H


def test_rht16_is_the_scaled_sylvester_product(orc):
    """Integer inputs: every butterfly sum is exact, so the oracle must give
    (1/4) H16 (s .* v) exactly (rational arithmetic)."""
    H = _sylvester16()
    rng = np.random.default_rng(31)
    for _ in range(200):
        v = rng.integers(-4096, 4096, 16)
        s = int(rng.integers(0, 1 << 16))
        sv = [Fraction(int(v[i]) * (-1 if (s >> i) & 1 else 1)) for i in range(16)]
        want = [sum(H[i, k] * sv[k] for k in range(16)) / 4 for i in range(16)]
        got = orc.rht16(v.astype(np.float32), s)
        assert [Fraction(float(g)) for g in got] == want


def test_rht16_is_orthonormal_and_its_own_inverse(orc):
    rng = np.random.default_rng(32)
    for _ in range(100):
        v = rng.integers(-1000, 1000, 16).astype(np.float32)
        s = int(rng.integers(0, 1 << 16))
        back = orc.rht16(orc.rht16(v, s), 0)              # (H/4)(H/4) = I, then undo the signs
        flip = np.array([-1 if (s >> i) & 1 else 1 for i in range(16)], np.float32)
        assert (back * flip == v).all()
        w = rng.standard_normal(16).astype(np.float32) * np.float32(10.0 ** rng.uniform(-20, 20))
        z = orc.rht16(w, s).astype(np.float64)
        nw = np.linalg.norm(w.astype(np.float64))
        assert abs(np.linalg.norm(z) - nw) <= 1e-6 * nw


def test_rht16_overflow_is_sanitized(orc):
    big = np.full(16, np.float32(3.3895314e38))            # largest finite bf16
    z = orc.rht16(big, 0, in_dtype="bf16")
    assert np.isfinite(z).all()
    assert z[0] == np.float32(3.3895314e38) and (z[1:] == 0).all()


def test_col_hadamard_quantize_is_quantize_of_the_transform(orc):
    """With col_hadamard, the columnwise codes and scales are those of the
    ordinary columnwise quantization of the transformed tensor; the rowwise
    side is untouched."""
    x = W.lognormal((1, 64, 64), 34, sigma=2.0)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xf = x.float().numpy()[0]
    s = 0xA5C3
    z = np.empty_like(xf)
    for j in range(64):
        for i0 in range(0, 64, 16):
            z[i0:i0 + 16, j] = orc.rht16(xf[i0:i0 + 16, j], s, in_dtype="bf16")
    for kw in (dict(mode="none"), dict(mode="outer_block", ob=16), dict(mode="outer_block", ob=32),
               dict(mode="none", rounding="sr", seed=4, step=1)):
        got = orc.quantize(xb, out_mask=3, col_hadamard=True, hadamard_signs=s, **kw)
        ref_row = orc.quantize(xb, out_mask=1, **kw)
        ref_col = orc.quantize(z[None].astype(np.float32), out_mask=2, **kw)
        assert (got["row_codes"] == ref_row["row_codes"]).all() and (got["row_scales"] == ref_row["row_scales"]).all()
        assert (got["col_codes"] == ref_col["col_codes"]).all() and (got["col_scales"] == ref_col["col_scales"]).all()
        if kw["mode"] == "outer_block":
            assert (got["col_outer"].view(np.uint32) == ref_col["col_outer"].view(np.uint32)).all()


# ----------------------------------------------------------------------------
# input sanitization (reading Q6 of "NaN-input sanitization")
# ----------------------------------------------------------------------------

BF16_MAX = bits_f32(0x7F7F0000)
F32_MAX = float(np.finfo(np.float32).max)


def _plant_nonfinite(x_f32, rng):
    """Scatter NaN (both signs), +inf and -inf over x (binary32 values);
    returns the positions of each kind."""
    n = x_f32.size
    pos = rng.permutation(n)[:4 * 12].reshape(4, 12)
    flat = x_f32.reshape(-1)
    flat[pos[0]] = np.float32(np.nan)
    flat[pos[1]] = -np.float32(np.nan)
    flat[pos[2]] = np.float32(np.inf)
    flat[pos[3]] = -np.float32(np.inf)
    return pos


def _as_input(xf, dtype):
    if dtype == "fp32":
        return np.ascontiguousarray(xf, np.float32)
    return bf16_np(torch.from_numpy(np.ascontiguousarray(xf, np.float32)).to(torch.bfloat16))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("kw", [dict(mode="none"), dict(mode="tensorwise"), dict(mode="outer_block", ob=32),
                                dict(mode="outer_block", ob=32, outer_2d=True),
                                dict(mode="outer_block", ob=16, inner_2d=True)],
                         ids=["none", "tensorwise", "ob32", "ob32-2d", "ob16-in2d"])
def test_nonfinite_inputs_read_as_sanitized_values(orc, dtype, kw):
    """ALTO "Op-level test coverage" names NaN-input sanitization without its
    rule; the reading is NaN -> +0 and +-inf -> +- the largest finite value of
    the input dtype, before any amax.  A tensor holding NaN / +inf / -inf must
    quantize, in both orientations, exactly like the same tensor with +0,
    +max and -max written in those places (max = 0x7F7F in bf16, FLT_MAX in
    binary32), error-feedback residual included.  A NaN read as -0, the
    binary32 maximum used for bf16 input, or a non-finite value reaching an
    amax all break the equality."""
    rng = np.random.default_rng(40)
    xf = rng.standard_normal((64, 96)).astype(np.float32)
    pos = _plant_nonfinite(xf, rng)
    mx = BF16_MAX if dtype == "bf16" else F32_MAX
    xs = xf.copy().reshape(-1)
    xs[pos[0]] = 0.0
    xs[pos[1]] = 0.0
    xs[pos[2]] = mx
    xs[pos[3]] = -mx
    a, b = _as_input(xf, dtype), _as_input(xs.reshape(64, 96), dtype)
    assert not np.array_equal(a, b)
    qa = orc.quantize(a, out_mask=3, **kw)
    qb = orc.quantize(b, out_mask=3, **kw)
    for k, v in qa.items():
        if v is not None:
            np.testing.assert_array_equal(v.view(np.uint8), qb[k].view(np.uint8), err_msg=k)
    # error feedback: u = sanitize(x + r) with r = 0, residual u - deq finite
    ra = np.zeros((1, 64, 96), np.float32)
    rb = np.zeros((1, 64, 96), np.float32)
    orc.quantize(a, residual=ra, **kw)
    orc.quantize(b, residual=rb, **kw)
    assert np.all(np.isfinite(ra))
    np.testing.assert_array_equal(ra.view(np.uint32), rb.view(np.uint32))


@pytest.mark.parametrize("dtype,mx", [("bf16", BF16_MAX), ("fp32", F32_MAX)])
def test_nonfinite_inputs_closed_form(orc, dtype, mx):
    """The same reading written out on one 1 x 16 block per case.
    Mode none: the block [NaN, +inf, -inf, 1, 0 ...] has amax = max (the
    sanitized infinity), so the inner scale saturates at 448 (code 0x7E); the
    NaN becomes code 0x0 (+0, not 0x8), +-inf code 0x7 / 0xF (+-6), and 1/448
    rounds to +0.  Tensorwise: the scale is max / 2688 in binary32, which
    tells the bf16 maximum from the binary32 one."""
    xf = np.zeros((1, 16), np.float32)
    xf[0, :4] = [np.nan, np.inf, -np.inf, 1.0]
    x = _as_input(xf, dtype)
    q = orc.quantize(x, mode="none")
    assert q["row_scales"][0, 0, 0] == 0x7E
    codes = _unpack(q["row_codes"])[0, 0]
    assert list(codes[:4]) == [0x0, 0x7, 0xF, 0x0]
    assert set(codes[4:]) == {0x0}
    t = orc.quantize(x, mode="tensorwise")
    want = np.float32(mx) / np.float32(2688.0)
    assert t["tile_outer"][0].view(np.uint32) == want.view(np.uint32)
    # a block of NaNs alone: every value +0, amax 0, scale 0, codes +0
    z = _as_input(np.full((1, 16), np.nan, np.float32), dtype)
    qz = orc.quantize(z, mode="tensorwise")
    assert qz["tile_outer"][0] == 0.0 and not np.signbit(qz["tile_outer"][0])
    assert qz["row_scales"][0, 0, 0] == 0 and set(_unpack(qz["row_codes"])[0, 0]) == {0x0}


# ----------------------------------------------------------------------------
# inner scales in the tensor-core layout (NVIDIA's published block-scaling-
# factor layout, read by block-scaled FP4 MMAs)
# ----------------------------------------------------------------------------

def test_scale_layout_mma_worked_positions(orc):
    """Positions the cuBLAS description of the 128 x 4 block layout fixes:
    within a 512-byte block, row r and column c go to 16 (r mod 32) +
    4 (r div 32) + c; blocks follow in row-major order of (row block,
    column block); a second matrix starts after the first one's blocks."""
    G, R, C = 2, 200, 9            # 2 row blocks x 3 column blocks per matrix
    lin = np.zeros((G, R, C), np.uint8)
    want = {}
    for (g, r, c), off in {(0, 0, 0): 0, (0, 0, 1): 1, (0, 1, 0): 16, (0, 31, 3): 16 * 31 + 3, (0, 32, 0): 4,
                           (0, 96, 2): 14, (0, 127, 3): 511, (0, 0, 4): 512, (0, 0, 8): 1024,
                           (0, 128, 0): 3 * 512, (0, 199, 5): 4 * 512 + 16 * (71 % 32) + 4 * (71 // 32) + 1,
                           (1, 0, 0): 6 * 512, (1, 33, 6): 6 * 512 + 1 * 512 + 16 + 4 + 2}.items():
        lin[g, r, c] = len(want) + 1
        want[off] = len(want) + 1
    out = orc.scale_layout_mma(lin)
    assert out.size == G * 2 * 3 * 512
    assert {int(i): int(out[i]) for i in np.flatnonzero(out)} == want


def test_scale_layout_mma_is_a_zero_padded_permutation(orc):
    """Every scale byte lands in exactly one place and every padding byte is
    zero; the layout agrees with an independent formulation of the same
    description (pad, cut into 128 x 4 blocks, interleave the four 32-row
    groups of a block) written with array reshapes."""
    from gpu_helpers import to_mma_layout

    rng = np.random.default_rng(41)
    for G, R, C in ((1, 128, 4), (2, 208, 20), (1, 33, 3), (3, 256, 180), (1, 5760, 180)):
        lin = rng.integers(1, 256, size=(G, R, C), dtype=np.uint8)
        out = orc.scale_layout_mma(lin)
        assert out.size == G * (-(-R // 128)) * (-(-C // 4)) * 512
        assert np.count_nonzero(out) == lin.size
        assert np.array_equal(np.sort(out[out != 0]), np.sort(lin.ravel()))
        np.testing.assert_array_equal(out, to_mma_layout(lin))
