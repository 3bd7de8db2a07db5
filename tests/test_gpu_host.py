"""mxfp4_fake_quantize_host: the host-buffer entry point streams chunks of
rows through the GPU; its output must equal the device entry point's (and so
the oracle's, which the device path is tested against) bit for bit, for
single and many chunks, ragged last chunks, strided host views, both dtypes,
pinned and pageable memory."""
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import host_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


def _same(a: torch.Tensor, b: torch.Tensor):
    assert a.shape == b.shape and a.dtype == b.dtype
    assert (host_np(a) == host_np(b)).all() if a.dtype == torch.bfloat16 else \
        (host_np(a).view("u4") == host_np(b).view("u4")).all()


@pytest.mark.parametrize("pinned", [True, False])
def test_host_matches_device_headline_rows(pinned):
    x, _ = W.mxfp4_weight()
    x = x[:3000]  # 3000 x 8192 bf16 = 49 MB: several chunks, a ragged last one
    xh = x.pin_memory() if pinned else x
    y = fq.mxfp4_fake_quantize_host(xh)
    _same(y, fq.mxfp4_fake_quantize(x.cuda()).cpu())


def test_host_many_small_chunks_and_strided_view():
    base = W.lognormal((2, 96, 320), 51, sigma=3.0).pin_memory()
    xv = base[:, :, 32:288]  # K = 256, row stride 320, in pinned memory
    ws = torch.empty(2 * (512 + 512) + 2 * (6 * 512 + 6 * 512), dtype=torch.uint8, device="cuda")  # a few rows per chunk
    assert xv.stride(1) == 320
    y = fq.mxfp4_fake_quantize_host(xv, workspace=ws)
    _same(y, fq.mxfp4_fake_quantize(xv.contiguous().cuda()).cpu())


@pytest.mark.parametrize("din,dout", [(torch.float32, torch.float32), (torch.bfloat16, torch.float32),
                                      (torch.float32, torch.bfloat16)])
def test_host_dtypes(din, dout):
    x = W.lognormal((1, 257, 512), 52, sigma=4.0, dtype=din)
    x.view(-1)[100] = float("nan")
    y = fq.mxfp4_fake_quantize_host(x.pin_memory(), out_dtype=dout)
    _same(y, fq.mxfp4_fake_quantize(x.cuda(), out_dtype=dout).cpu())


def test_host_rejects_small_workspace_and_device_input():
    x = W.lognormal((1, 16, 64), 53).pin_memory()
    with pytest.raises(fq.FP4QError):
        fq.mxfp4_fake_quantize_host(x, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError):
        fq.mxfp4_fake_quantize_host(x.cuda())
