"""The row-sharded path on one GPU: each shard's amax from fp4_tensor_amax,
their maximum, then each shard quantized with the shared tensorwise scale
(the single-process stand-in for the all-reduce) gives exactly the slices
of the unsharded result; outer-block modes shard with no exchange."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import sharded
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import host_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


def _np_amax(x: torch.Tensor, in_dtype) -> np.float32:
    """max |x| after the sanitizing rule: NaN -> 0, inf -> the largest finite
    value of the input dtype."""
    a = np.abs(x.float().cpu().numpy())
    a[np.isnan(a)] = 0.0
    a[np.isinf(a)] = float(torch.finfo(in_dtype).max)
    return np.float32(a.max() if a.size else 0.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tensor_amax_matches_definition(dtype):
    x = W.lognormal((3, 96, 208), 41, sigma=2.0, dtype=dtype)
    x.view(-1)[11] = float("nan")
    x.view(-1)[999] = float("-inf")
    a = fq.tensor_amax(x.cuda())
    assert a.cpu().numpy().view(np.uint32)[0] == _np_amax(x, dtype).view(np.uint32)
    r = torch.randn(3, 96, 208, generator=torch.Generator("cpu").manual_seed(3)) * 1e3
    a2 = fq.tensor_amax(x.cuda(), residual=r.cuda())
    u = x.float() + r  # binary32, round to nearest
    assert a2.cpu().numpy().view(np.uint32)[0] == _np_amax(u, dtype).view(np.uint32)
    assert fq.tensor_amax(torch.empty(0, 64, dtype=dtype, device="cuda")).item() == 0.0


@pytest.mark.parametrize("columnwise", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "ue5m3"])
def test_tensorwise_shards_equal_unsharded(columnwise, fmt):
    x = W.activations(M=1024, K=512, n_cols=3, n_rows=2).cuda()
    kw = dict(rowwise=True, columnwise=columnwise, scale_format=fmt)
    full = fq.quantize(x, mode="tensorwise", **kw)
    world = 3
    align = sharded.shard_alignment("tensorwise", columnwise=columnwise)
    parts = [sharded.row_range(x.shape[0], world, r, max(align, 128)) for r in range(world)]
    amax = torch.stack([fq.tensor_amax(x[lo:hi]) for lo, hi in parts]).max().reshape(1)
    S = sharded.tensorwise_scale(amax, fmt)
    assert torch.equal(S.view(torch.int32), full.tile_outer.view(torch.int32))
    for lo, hi in parts:
        pre = fq.QuantizedFP4((1, hi - lo, 512), "tensorwise", 0, False, False, fmt, tile_outer=S)
        q = fq.quantize(x[lo:hi], mode="tensorwise", precomputed_outer=pre, **kw)
        assert torch.equal(q.row_codes[0], full.row_codes[0, lo:hi])
        assert torch.equal(q.row_scales[0], full.row_scales[0, lo:hi])
        if columnwise:
            assert torch.equal(q.col_codes[0], full.col_codes[0, :, lo // 2:hi // 2])
            assert torch.equal(q.col_scales[0], full.col_scales[0, :, lo // 16:hi // 16])


def test_outer_block_shards_need_no_exchange():
    x = W.activations(M=1024, K=512, n_cols=3, n_rows=2).cuda()
    kw = dict(mode="outer_block", outer_block_size=64, outer_2d=True, rowwise=True, columnwise=True)
    full = fq.quantize(x, **kw)
    align = sharded.shard_alignment("outer_block", 64, outer_2d=True, columnwise=True)
    for r in range(2):
        lo, hi = sharded.row_range(1024, 2, r, align)
        q = sharded.quantize_shard(x[lo:hi], **kw)
        assert torch.equal(q.row_codes[0], full.row_codes[0, lo:hi])
        assert torch.equal(q.col_codes[0], full.col_codes[0, :, lo // 2:hi // 2])
        assert torch.equal(q.tile_outer[0], full.tile_outer[0, lo // 64:hi // 64])
