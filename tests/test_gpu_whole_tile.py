"""The whole-tile form of the bf16 cast-transpose quantize (M a multiple of
128, K of 64, both orientations, round-to-nearest; no outer scale, one per
tensor, 1 x 64 / 64 x 1 or 64 x 64 outer blocks) against the oracle, bit for
bit, on data that keeps every warp on the fast sequences and on data that
sends warps to the general per-block steps (all-zero blocks, maxima below
2^-90, subnormals, non-finite inputs, values at the bf16 maximum), and
against the general cast-transpose kernel (FP4Q_NO_CTL_KERNEL=1)."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import assert_same, gpu_quantize, host_np, oracle_quantize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


MODES = {"none": dict(mode="none"), "tensorwise": dict(mode="tensorwise"),
         "ob64": dict(mode="outer_block", outer_block_size=64),
         "ob64-2d": dict(mode="outer_block", outer_block_size=64, outer_2d=True)}


def _special(shape, seed):
    """Lognormal data with planted blocks that leave the fast range."""
    x = W.lognormal(shape, seed, sigma=2.0).float()
    G, M, K = shape
    g = torch.Generator().manual_seed(seed + 1)
    flat = x.view(G, M, K)
    for _ in range(6):                                   # all-zero 16 x 16 patches
        r, c = int(torch.randint(0, M // 16, (1,), generator=g)) * 16, int(torch.randint(0, K // 16, (1,), generator=g)) * 16
        flat[0, r:r + 16, c:c + 16] = 0.0
    for _ in range(4):                                   # tiny patches (below 2^-90, some subnormal)
        r, c = int(torch.randint(0, M // 16, (1,), generator=g)) * 16, int(torch.randint(0, K // 16, (1,), generator=g)) * 16
        flat[-1, r:r + 16, c:c + 16] = torch.randn(16, 16, generator=g) * 2.0 ** -120
    flat[0, 64:128, 0:64] = torch.randn(64, 64, generator=g) * 2.0 ** -118   # a whole 64 x 64 block below 2^-90
    flat[0, 5, 7] = float("nan")
    flat[-1, M - 3, K - 9] = float("inf")
    flat[0, M // 2, 3] = -float("inf")
    flat[-1, 17, K // 2] = 3.3e38                        # rounds to the bf16 maximum
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("shape", [(1, 128, 64), (2, 256, 192), (1, 384, 320)], ids=["one-tile", "g2", "3x5"])
@pytest.mark.parametrize("data", ["lognormal", "special"])
def test_whole_tile_matches_oracle(orc, fmt, mode, shape, data, monkeypatch):
    x = W.lognormal(shape, 81, sigma=2.0) if data == "lognormal" else _special(shape, 82)
    kw = dict(MODES[mode], scale_format=fmt, rowwise=True, columnwise=True)
    _, g = gpu_quantize(x, **kw)
    assert_same(g, oracle_quantize(orc, x, **kw))
    monkeypatch.setenv("FP4Q_NO_CTL_KERNEL", "1")           # the general cast-transpose kernel
    _, g2 = gpu_quantize(x, **kw)
    assert_same(g2, {k: v for k, v in g.items() if v is not None})


def test_whole_tile_precomputed_scales(orc):
    """Tensorwise with a given scale and with a given amax; 2-D outer blocks
    with given scales."""
    x = W.lognormal((2, 256, 128), 83, sigma=1.5)
    xd = x.cuda()
    full = fq.quantize(xd, mode="tensorwise", rowwise=True, columnwise=True)
    pre = fq.quantize(xd, mode="tensorwise", rowwise=True, columnwise=True, precomputed_outer=full)
    ws = fq.tensorwise_workspace("cuda")
    fq.tensor_amax(xd, out=fq.workspace_amax(ws))
    amx = fq.quantize(xd, mode="tensorwise", rowwise=True, columnwise=True, tensorwise_amax=ws)
    for q in (pre, amx):
        for k in ("row_codes", "row_scales", "col_codes", "col_scales", "tile_outer"):
            assert torch.equal(getattr(q, k), getattr(full, k)), k
    kw = dict(mode="outer_block", outer_block_size=64, outer_2d=True, rowwise=True, columnwise=True)
    a = fq.quantize(xd, **kw)
    b = fq.quantize(xd, precomputed_outer=a, **kw)
    for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    assert_same({k: host_np(getattr(a, k)) for k in ("row_codes", "col_codes", "tile_outer")},
                oracle_quantize(orc, x, **kw), keys=["row_codes", "col_codes", "tile_outer"])


def test_whole_tile_reused_outputs_and_back_to_back_calls():
    """Back-to-back calls into the same buffers (the deferred column stores
    of one call complete before the next call's kernel starts)."""
    xs = [W.lognormal((1, 512, 256), 84 + i, sigma=2.0).cuda() for i in range(3)]
    kw = dict(mode="outer_block", outer_block_size=64, rowwise=True, columnwise=True)
    refs = [fq.quantize(x, **kw) for x in xs]
    torch.cuda.synchronize()
    q = fq.quantize(xs[0], **kw)
    for i in range(9):
        fq.quantize(xs[i % 3], out=q, **kw)
        if i % 3 == 2:
            torch.cuda.synchronize()
            r = refs[2]
            for k in ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer"):
                assert torch.equal(getattr(q, k), getattr(r, k)), k


# outer amax values at the edges of the pair-table range (bf16 values):
# 2^-90 and just above (the smallest S), the largest in range with sigma = 1
# (m = 40: the folded zl of S = 2^89 is exactly 2^-126) and with m = 127,
# and the first ones outside (the general steps)
_EDGES = {"e4m3": [2.0 ** -90, 1.0078125 * 2.0 ** -90, 1.3125 * 2.0 ** 100, 1.9921875 * 2.0 ** 100, 2.0 ** 101,
                   1.5 * 2.0 ** -91],
          "ue5m3": [2.0 ** -90, 1.3125 * 2.0 ** 108, 1.9921875 * 2.0 ** 108, 2.0 ** 109, 1.5 * 2.0 ** -91]}


def _edge_blocks(amaxes, seed):
    """[1, 128, 64 * n]: one 128 x 64 tile per amax, every 64 x 64 block and
    every 1 x 64 / 64 x 1 group of it holding that amax, the other values
    spread over 2^-30 of it up to it."""
    g = torch.Generator().manual_seed(seed)
    tiles = []
    for A in amaxes:
        t = torch.rand(128, 64, generator=g, dtype=torch.float64) * 2.0 - 1.0
        t = t * torch.pow(2.0, -30.0 * torch.rand(128, 64, generator=g, dtype=torch.float64))
        t = t * A
        idx = torch.arange(128)
        t[idx, (idx * 7) % 64] = A * torch.where(idx % 2 == 0, 1.0, -1.0).double()   # each row's max
        t[(torch.arange(64) * 5) % 128, torch.arange(64)] = A                          # each column's max
        tiles.append(t)
    return torch.cat(tiles, dim=1)[None].to(torch.bfloat16)


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
@pytest.mark.parametrize("mode,cols", [("ob64", True), ("ob64-2d", True), ("ob64", False)],
                         ids=["ob64", "ob64-2d", "ob64-rowwise"])
def test_whole_tile_scale_range_edges(orc, fmt, mode, cols, monkeypatch):
    """The whole-tile kernel (rowwise + columnwise) and the bulk rowwise
    kernel (rowwise only) on outer amax values at the pair table's range
    edges, against the oracle and against the general kernels."""
    x = _edge_blocks(_EDGES[fmt], 95)
    assert (x.float().abs().amax(dim=1)[0].view(-1, 64).amax(dim=1).double() ==
            torch.tensor(_EDGES[fmt], dtype=torch.float64)).all()
    kw = dict(MODES[mode], scale_format=fmt, rowwise=True, columnwise=cols)
    _, g = gpu_quantize(x, **kw)
    assert_same(g, oracle_quantize(orc, x, **kw))
    monkeypatch.setenv("FP4Q_NO_CTL_KERNEL", "1")
    monkeypatch.setenv("FP4Q_GENERAL_KERNEL", "1")
    _, g2 = gpu_quantize(x, **kw)
    assert_same(g2, {k: v for k, v in g.items() if v is not None})


@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
@pytest.mark.parametrize("cols", [True, False], ids=["both", "rowwise"])
def test_whole_tile_tensorwise_range_edges(orc, fmt, cols):
    for A in _EDGES[fmt]:
        x = _edge_blocks([A], 96)
        kw = dict(MODES["tensorwise"], scale_format=fmt, rowwise=True, columnwise=cols)
        _, g = gpu_quantize(x, **kw)
        assert_same(g, oracle_quantize(orc, x, **kw))
