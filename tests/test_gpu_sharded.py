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
    # each shard's amax into its workspace, then their maximum (the all-reduce)
    wss = [fq.tensorwise_workspace("cuda") for _ in parts]
    for ws, (lo, hi) in zip(wss, parts):
        fq.tensor_amax(x[lo:hi], out=fq.workspace_amax(ws))
    amax = torch.stack([fq.workspace_amax(ws) for ws in wss]).max()
    for ws in wss:
        fq.workspace_amax(ws).fill_(amax)
    for ws, (lo, hi) in zip(wss, parts):
        q = fq.quantize(x[lo:hi], mode="tensorwise", tensorwise_amax=ws, **kw)
        assert torch.equal(q.tile_outer.view(torch.int32), full.tile_outer.view(torch.int32))
        assert torch.equal(q.row_codes[0], full.row_codes[0, lo:hi])
        assert torch.equal(q.row_scales[0], full.row_scales[0, lo:hi])
        if columnwise:
            assert torch.equal(q.col_codes[0], full.col_codes[0, :, lo // 2:hi // 2])
            assert torch.equal(q.col_scales[0], full.col_scales[0, :, lo // 16:hi // 16])


def test_single_process_quantize_shard_is_the_whole_tensor():
    """quantize_shard with no process group: the shard is the tensor, and the
    tensorwise scale comes from the device-side division of its amax."""
    x = W.lognormal((256, 384), 44, sigma=2.0).cuda()
    for fmt in ("e4m3", "ue5m3"):
        a = sharded.quantize_shard(x, mode="tensorwise", scale_format=fmt, rowwise=True, columnwise=True)
        b = fq.quantize(x, mode="tensorwise", scale_format=fmt, rowwise=True, columnwise=True)
        for k in ("row_codes", "row_scales", "col_codes", "col_scales"):
            assert torch.equal(getattr(a, k), getattr(b, k)), k
        assert torch.equal(a.tile_outer.view(torch.int32), b.tile_outer.view(torch.int32))


@pytest.mark.parametrize("kw", [dict(mode="none"), dict(mode="outer_block", outer_block_size=64),
                                dict(mode="tensorwise"), dict(mode="outer_block", outer_block_size=32, outer_2d=True)],
                         ids=["none", "ob64", "tensorwise", "ob32-2d"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_stochastic_rounding_shards_equal_unsharded(kw, dtype):
    """fp4-train README, "Method": the SR draw is keyed on (seed, step,
    global-index).  Row shards that pass their global row offset draw the
    words of the unsharded tensor, so their rowwise and columnwise codes are
    slices of the unsharded SR result."""
    M, K = 768, 320
    x = W.lognormal((M, K), 45, sigma=1.5, dtype=dtype).cuda()
    tw = kw["mode"] == "tensorwise"
    if tw:  # one process here: the whole tensor's amax stands for the all-reduced one
        ws = fq.tensorwise_workspace("cuda")
        fq.tensor_amax(x, out=fq.workspace_amax(ws))
    for columnwise in (True, False):
        q_kw = dict(kw, rowwise=True, columnwise=columnwise, stochastic=True, seed=0x1234_5678_9ABC, step=17)
        full = fq.quantize(x, **q_kw)
        align = sharded.shard_alignment(kw["mode"], kw.get("outer_block_size", 0), kw.get("outer_2d", False),
                                        columnwise=columnwise)
        for world in (2, 3):
            for r in range(world):
                lo, hi = sharded.row_range(M, world, r, max(align, 64))
                if tw:
                    q = fq.quantize(x[lo:hi], tensorwise_amax=ws, sr_global_rows=M, sr_row_offset=lo, **q_kw)
                else:
                    q = sharded.quantize_shard(x[lo:hi], row_offset=lo, global_rows=M, **q_kw)
                assert torch.equal(q.row_codes[0], full.row_codes[0, lo:hi]), (world, r)
                assert torch.equal(q.row_scales[0], full.row_scales[0, lo:hi])
                if columnwise:
                    assert torch.equal(q.col_codes[0], full.col_codes[0, :, lo // 2:hi // 2]), (world, r)
                    assert torch.equal(q.col_scales[0], full.col_scales[0, :, lo // 16:hi // 16])
                # without the global index the shard draws other words
                if world == 2 and r == 1 and not tw:
                    q2 = fq.quantize(x[lo:hi], **q_kw)
                    assert not torch.equal(q2.row_codes[0], full.row_codes[0, lo:hi])


def test_stochastic_rounding_expert_shards_equal_unsharded():
    """A stack of matrices sharded by matrix (experts across processes):
    sr_matrix_offset gives each shard the draws of its matrices in the
    whole stack, rowwise and columnwise."""
    x = W.moe_experts(G=4, M=128, K=192, experts=[0, 1, 2, 3]).cuda()
    q_kw = dict(mode="outer_block", outer_block_size=64, outer_2d=True, rowwise=True, columnwise=True,
                stochastic=True, seed=5, step=2)
    full = fq.quantize(x, **q_kw)
    for g0, g1 in ((0, 1), (1, 3), (3, 4)):
        q = fq.quantize(x[g0:g1], sr_matrix_offset=g0, **q_kw)
        for k in ("row_codes", "row_scales", "col_codes", "col_scales", "tile_outer"):
            assert torch.equal(getattr(q, k), getattr(full, k)[g0:g1]), (g0, k)


def test_stochastic_rounding_qdq_shard_with_error_feedback():
    """The SR + error-feedback QDQ of a row shard equals the rows of the
    whole-tensor QDQ (outputs and residuals), fp32 weight."""
    M, K = 512, 256
    w = (torch.randn(M, K, generator=torch.Generator().manual_seed(46)) * 0.02).cuda()
    r_full = (torch.randn(M, K, generator=torch.Generator().manual_seed(47)) * 1e-4).cuda()
    r_part = r_full.clone()
    y_full, _ = fq.qdq(w, mode="none", stochastic=True, seed=9, step=4, residual=r_full, out_dtype=torch.float32)
    for lo, hi in ((0, 192), (192, 512)):
        rp = r_part[lo:hi].contiguous()
        y, _ = fq.qdq(w[lo:hi], mode="none", stochastic=True, seed=9, step=4, residual=rp, out_dtype=torch.float32,
                      sr_global_rows=M, sr_row_offset=lo)
        assert torch.equal(y.view(torch.int32), y_full[lo:hi].view(torch.int32))
        assert torch.equal(rp.view(torch.int32), r_full[lo:hi].view(torch.int32))


def test_stochastic_rounding_shard_matches_oracle(orc):
    """One shard's SR codes against the oracle's codes of the whole tensor
    (the oracle quantizes the whole tensor; the shard is its row slice)."""
    M, K = 256, 128
    x = W.lognormal((M, K), 48, sigma=1.0)
    lo, hi = 64, 192
    q = fq.quantize(x[lo:hi].cuda(), rowwise=True, columnwise=True, stochastic=True, seed=3, step=1,
                    sr_global_rows=M, sr_row_offset=lo)
    r = orc.quantize(host_np(x)[None], out_mask=3, rounding="sr", seed=3, step=1)
    assert (host_np(q.row_codes[0]) == r["row_codes"][0, lo:hi]).all()
    assert (host_np(q.col_codes[0]) == r["col_codes"][0, :, lo // 2:hi // 2]).all()


def test_precomputed_amax_qdq():
    """QDQ with the tensorwise amax supplied: the same outputs and scale as
    the QDQ that computes it."""
    x = W.lognormal((2, 128, 256), 49, sigma=2.0).cuda()
    y0, s0 = fq.qdq(x, mode="tensorwise", out_dtype=torch.float32)
    ws = fq.tensorwise_workspace("cuda")
    fq.tensor_amax(x, out=fq.workspace_amax(ws))
    y1, s1 = fq.qdq(x, mode="tensorwise", out_dtype=torch.float32, tensorwise_amax=ws)
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    assert torch.equal(s0.view(torch.int32), s1.view(torch.int32))


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
