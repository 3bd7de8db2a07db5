"""Fused MXFP4 projection + MXFP8 re-encode against the oracle, bit for bit:
all bf16 patterns, the headline weight's edge blocks, fp32 inputs, ragged
tiles and batches; the projection output equals mxfp4_fake_quantize's."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import assert_same, host_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


@pytest.fixture(params=["tma", "plain"], autouse=True)
def form(request, monkeypatch):
    """bf16 input takes the persistent TMA-fed kernel; "plain" forces the
    one-tile-per-CTA kernel (fp32 input always takes it)."""
    monkeypatch.delenv("FP4Q_NO_MX8_TMA", raising=False)
    if request.param == "plain":
        monkeypatch.setenv("FP4Q_NO_MX8_TMA", "1")
    return request.param


def _check(orc, x, rowwise=True, columnwise=True, out_dtype=None):
    out_dtype = out_dtype or x.dtype
    q = fq.mxfp4_project_mxfp8(x.cuda(), rowwise=rowwise, columnwise=columnwise, with_y=True, out_dtype=out_dtype)
    torch.cuda.synchronize()
    xo = host_np(x)
    ref = orc.mxfp4_project_mxfp8(xo if xo.ndim == 3 else xo[None],
                                  out_dtype="bf16" if out_dtype == torch.bfloat16 else "fp32",
                                  out_mask=(1 if rowwise else 0) | (2 if columnwise else 0))
    got = {k: host_np(getattr(q, k)) for k in ("y", "row_codes", "row_scales", "col_codes", "col_scales")
           if getattr(q, k) is not None}
    assert_same(got, ref)
    yd = fq.mxfp4_fake_quantize(x.cuda(), out_dtype=out_dtype)
    assert torch.equal(q.y.reshape(yd.shape).view(torch.uint8), yd.view(torch.uint8))


def test_all_bf16_patterns(orc):
    _check(orc, W.all_bf16_patterns())


def test_headline_rows_with_edge_blocks(orc):
    x, _ = W.mxfp4_weight()
    _check(orc, x[:1024, :4096])


@pytest.mark.parametrize("shape", [(1, 160, 96), (2, 64, 224), (1, 32, 32)], ids=["ragged", "batch", "one-tile"])
@pytest.mark.parametrize("din,dout", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                      (torch.float32, torch.bfloat16)])
def test_shapes_and_dtypes(orc, shape, din, dout):
    x = W.lognormal(shape, 81, sigma=6.0, dtype=din)
    x.view(-1)[3] = float("inf")
    _check(orc, x, out_dtype=dout)


def test_rowwise_only_any_rows(orc):
    x = W.lognormal((1, 100, 64), 82, sigma=3.0)
    _check(orc, x, columnwise=False)
    with pytest.raises(fq.FP4QError):
        fq.mxfp4_project_mxfp8(x.cuda(), columnwise=True)  # M % 32 != 0


def test_more_tiles_than_resident_ctas(orc):
    # 2 x 16 x 33 = 1056 tiles of 128 x 64, more than one wave of resident
    # CTAs, with a half-filled last tile column
    x = W.lognormal((2, 2048, 2080), 83, sigma=4.0)
    _check(orc, x)


def test_outputs_16_bytes_past_a_32_byte_boundary(orc):
    """Projection and rowwise codes 16 bytes past a 32-byte boundary take the
    16-byte stores (32-byte aligned ones the 256-bit stores); same bits."""
    G, M, K = 1, 96, 256
    x = W.lognormal((G, M, K), 84, sigma=4.0)
    n = G * M * K
    ybuf = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    cbuf = torch.empty(n + 32, dtype=torch.uint8, device="cuda")
    out = fq.MXFP8Pair()
    out.y = ybuf[8:8 + n].view(G, M, K)
    out.row_codes = cbuf[16:16 + n].view(G, M, K)
    out.row_scales = torch.empty(G, M, K // 32, dtype=torch.uint8, device="cuda")
    assert out.y.data_ptr() % 32 == 16 and out.row_codes.data_ptr() % 32 == 16
    q = fq.mxfp4_project_mxfp8(x.cuda(), columnwise=False, with_y=True, out=out)
    ref = orc.mxfp4_project_mxfp8(host_np(x), out_dtype="bf16", out_mask=1)
    assert_same({k: host_np(getattr(q, k)) for k in ("y", "row_codes", "row_scales")},
                {k: ref[k] for k in ("y", "row_codes", "row_scales")})
