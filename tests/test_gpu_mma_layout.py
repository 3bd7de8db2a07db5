"""Inner scales in the tensor-core (128 x 4 tiled) layout: every kernel path
writes the same bytes as the linear layout rearranged by the layout's
definition (padding zero), codes unchanged; dequantize reads the layout; and
NVFP4 GEMMs in torch (cuBLASLt) consume codes and scales as written."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import host_np, to_mma_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


@pytest.fixture(params=["fast", "tile", "general"])
def kernel(request, monkeypatch):
    for v in ("FP4Q_GENERAL_KERNEL", "FP4Q_NO_ROW_KERNEL", "FP4Q_NO_CTB_KERNEL"):
        monkeypatch.delenv(v, raising=False)
    if request.param == "general":
        monkeypatch.setenv("FP4Q_GENERAL_KERNEL", "1")
    elif request.param == "tile":
        monkeypatch.setenv("FP4Q_NO_ROW_KERNEL", "1")
        monkeypatch.setenv("FP4Q_NO_CTB_KERNEL", "1")
    return request.param


CASES = [dict(mode="none"), dict(mode="tensorwise"), dict(mode="outer_block", outer_block_size=64),
         dict(mode="outer_block", outer_block_size=32, outer_2d=True), dict(mode="none", inner_2d=True),
         dict(mode="none", stochastic=True, seed=3)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(1, 208, 320), (2, 256, 448), (1, 96, 64)], ids=["pad-rows", "g2", "small"])
@pytest.mark.parametrize("case", CASES, ids=["none", "tensorwise", "ob64", "ob32-2d", "inner2d", "sr"])
def test_mma_layout_equals_rearranged_linear(case, shape, dtype, kernel):
    G, M, K = shape
    ob = case.get("outer_block_size", 0)
    if ob and (K % ob or M % ob):
        pytest.skip("shape not divisible by the outer block")
    x = W.lognormal(shape, 61, sigma=3.0, dtype=dtype).cuda()
    for mask in ((True, False), (False, True), (True, True)):
        kw = dict(case, rowwise=mask[0], columnwise=mask[1])
        lin = fq.quantize(x, **kw)
        mma = fq.quantize(x, scale_layout="mma", **kw)
        for o in ("row", "col"):
            if getattr(lin, o + "_codes") is None:
                continue
            assert torch.equal(getattr(mma, o + "_codes"), getattr(lin, o + "_codes"))
            want = to_mma_layout(host_np(getattr(lin, o + "_scales")))
            got = host_np(getattr(mma, o + "_scales"))
            assert got.shape == want.shape and (got == want).all(), (o, kw)
            y_lin = fq.dequantize(lin, o, torch.float32)
            y_mma = fq.dequantize(mma, o, torch.float32)
            assert torch.equal(y_lin.view(torch.int32), y_mma.view(torch.int32))


def test_mma_layout_padding_is_zero_on_reused_buffers():
    """Padding bytes are cleared by every call, also in a reused buffer."""
    x = W.lognormal((1, 208, 336), 62, sigma=2.0).cuda()
    q = fq.quantize(x, scale_layout="mma", rowwise=True, columnwise=True)
    q.row_scales.fill_(0xAB)
    q.col_scales.fill_(0xCD)
    fq.quantize(x, scale_layout="mma", rowwise=True, columnwise=True, out=q)
    lin = fq.quantize(x, rowwise=True, columnwise=True)
    assert (host_np(q.row_scales) == to_mma_layout(host_np(lin.row_scales))).all()
    assert (host_np(q.col_scales) == to_mma_layout(host_np(lin.col_scales))).all()


def _scaled_mm_nvfp4(a_codes, a_scales, b_codes, b_scales):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no float4_e2m1fn_x2")
    A = a_codes.view(torch.float4_e2m1fn_x2)
    B = b_codes.view(torch.float4_e2m1fn_x2)
    try:
        return torch._scaled_mm(A, B.t(), a_scales.view(torch.float8_e4m3fn), b_scales.view(torch.float8_e4m3fn),
                                out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip("torch._scaled_mm has no NVFP4 path here: %s" % str(e).splitlines()[0][:120])


@pytest.mark.parametrize("mnk", [(256, 384, 512), (208, 128, 320)], ids=["aligned", "padded"])
def test_nvfp4_gemm_reads_the_layout(mnk):
    """A block-scaled FP4 GEMM (cuBLASLt through torch) reads our codes and
    MMA-layout scales: its result equals the product of the dequantized
    operands up to binary32 accumulation order and the bf16 output rounding.
    A misplaced scale would change results by factors of 2 or more."""
    M, N, K = mnk
    a = W.lognormal((M, K), 63, sigma=2.0).cuda()
    b = W.lognormal((N, K), 64, sigma=2.0).cuda()
    qa = fq.quantize(a, scale_layout="mma")
    qb = fq.quantize(b, scale_layout="mma")
    y = _scaled_mm_nvfp4(qa.row_codes[0], qa.row_scales, qb.row_codes[0], qb.row_scales)
    da = fq.dequantize(qa, "row", torch.float32)[0].double()
    db = fq.dequantize(qb, "row", torch.float32)[0].double()
    ref = da @ db.t()
    err = (y.double() - ref).abs()
    tol = 1e-2 * (da.abs() @ db.abs().t()) + 1e-30
    assert (err <= tol).all(), float((err / tol).max())
