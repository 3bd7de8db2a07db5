"""Ragged grouped quantize against the oracle run on each group as a matrix
of its own (stochastic-rounding index base = the group's first flat index),
for every mode, mask and both scale formats, with empty and ragged groups;
invalid offsets write nothing and raise the workspace flag."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import assert_same, host_np, oracle_kw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


def _oracle_group(orc, xg, base, kw, mask):
    ok = oracle_kw(kw)
    m = (1 if mask[0] else 0) | (2 if mask[1] else 0)
    return orc.quantize(host_np(xg)[None], out_mask=m, sr_index_base=base, **ok)


CASES = [dict(mode="none"), dict(mode="tensorwise"), dict(mode="outer_block", outer_block_size=64),
         dict(mode="outer_block", outer_block_size=16, scale_format="ue5m3"),
         dict(mode="outer_block", outer_block_size=64, outer_2d=True), dict(mode="none", stochastic=True, seed=9)]


@pytest.fixture(params=["whole", "general"])
def kernel(request, monkeypatch):
    """Ragged groups with 64-row outer blocks and both orientations take the
    whole-tile kernel (half tiles at group tails); "general" forces the
    general cast-transpose kernel for the same calls."""
    monkeypatch.delenv("FP4Q_NO_CTL_KERNEL", raising=False)
    if request.param == "general":
        monkeypatch.setenv("FP4Q_NO_CTL_KERNEL", "1")
    return request.param


@pytest.mark.parametrize("case", CASES, ids=["none", "tensorwise", "ob64", "ob16-ue5m3", "ob64-2d", "sr"])
@pytest.mark.parametrize("mask", [(True, False), (False, True), (True, True)], ids=["row", "col", "both"])
def test_grouped_matches_per_group_oracle(orc, case, mask, kernel):
    if kernel == "general" and not (mask == (True, True) and case.get("outer_block_size") == 64):
        pytest.skip("the same kernel runs either way")
    align = 64 if case.get("outer_block_size", 0) == 64 else 16
    sizes = [0, 3 * align, 128, align, 5 * align + 128, 0, 2 * align]
    K = 320
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    T = int(off[-1])
    x = W.lognormal((T, K), 71, sigma=2.5)
    x.view(-1)[17] = float("nan")
    kw = dict(case, rowwise=mask[0], columnwise=mask[1])
    q = fq.quantize_grouped(x.cuda(), torch.from_numpy(off).cuda(), **kw)
    torch.cuda.synchronize()
    assert int(q.group_error.item()) == 0
    g = {k: (None if getattr(q, k) is None else host_np(getattr(q, k)))
         for k in ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer")}
    ob = case.get("outer_block_size", 0)
    for e in range(len(sizes)):
        a, b = int(off[e]), int(off[e + 1])
        if b == a:
            if case["mode"] == "tensorwise":
                assert g["tile_outer"].reshape(-1)[e] == 0.0
            continue
        r = _oracle_group(orc, x[a:b], a * K, kw, mask)
        got = {}
        if mask[0]:
            got["row_codes"] = g["row_codes"][0, a:b]
            got["row_scales"] = g["row_scales"][0, a:b]
            if r.get("row_outer") is not None:
                got["row_outer"] = g["row_outer"].reshape(T, -1)[a:b]
        if mask[1]:
            got["col_codes"] = g["col_codes"][K * a // 2:K * b // 2]
            got["col_scales"] = g["col_scales"][K * a // 16:K * b // 16]
            if r.get("col_outer") is not None:
                got["col_outer"] = g["col_outer"][K * a // ob:K * b // ob]
        if case["mode"] == "tensorwise":
            got["tile_outer"] = g["tile_outer"].reshape(-1)[e:e + 1]
        elif case.get("outer_2d"):
            got["tile_outer"] = g["tile_outer"].reshape(T // ob, K // ob)[a // ob:b // ob]
        keys = [k for k in got if r.get(k) is not None]
        assert_same(got, r, keys)


def test_grouped_invalid_offsets_write_nothing():
    x = W.lognormal((96, 128), 72).cuda()
    off = torch.tensor([0, 40, 96], dtype=torch.int64, device="cuda")  # 40 is not a multiple of 16
    q = fq.quantize_grouped(x, off, rowwise=True, columnwise=True)
    q.col_codes.fill_(0x5A)
    q.row_codes.fill_(0x5A)
    q = fq.quantize_grouped(x, off, rowwise=True, columnwise=True, out=q)
    torch.cuda.synchronize()
    assert int(q.group_error.item()) != 0
    assert bool((q.col_codes == 0x5A).all()) and bool((q.row_codes == 0x5A).all())
    off2 = torch.tensor([0, 48, 90], dtype=torch.int64, device="cuda")  # does not end at M
    q2 = fq.quantize_grouped(x, off2, rowwise=True)
    torch.cuda.synchronize()
    assert int(q2.group_error.item()) != 0


@pytest.mark.parametrize("outer_2d", [False, True], ids=["1d", "2d"])
def test_grouped_invalid_offsets_write_nothing_whole_tile(outer_2d):
    x = W.lognormal((256, 128), 73).cuda()
    off = torch.tensor([0, 64, 160, 256], dtype=torch.int64, device="cuda")  # 96 rows: not a multiple of 64
    kw = dict(mode="outer_block", outer_block_size=64, outer_2d=outer_2d, rowwise=True, columnwise=True)
    q = fq.quantize_grouped(x, off, **kw)
    for t in (q.col_codes, q.row_codes, q.col_scales, q.row_scales):
        t.fill_(0x5A)
    q = fq.quantize_grouped(x, off, out=q, **kw)
    torch.cuda.synchronize()
    assert int(q.group_error.item()) != 0
    for t in (q.col_codes, q.row_codes, q.col_scales, q.row_scales):
        assert bool((t == 0x5A).all())


def test_grouped_single_group_equals_plain_quantize():
    x = W.activations(M=1024, K=576, n_cols=3, n_rows=2).cuda()
    off = torch.tensor([0, 1024], dtype=torch.int64, device="cuda")
    for kw in (dict(mode="outer_block", outer_block_size=64), dict(mode="tensorwise"), dict(mode="none")):
        a = fq.quantize(x, rowwise=True, columnwise=True, **kw)
        b = fq.quantize_grouped(x, off, rowwise=True, columnwise=True, **kw)
        assert torch.equal(a.row_codes, b.row_codes) and torch.equal(a.row_scales, b.row_scales)
        assert torch.equal(a.col_codes.reshape(-1), b.col_codes) and torch.equal(a.col_scales.reshape(-1), b.col_scales)
        if kw["mode"] == "tensorwise":
            assert torch.equal(a.tile_outer, b.tile_outer)
