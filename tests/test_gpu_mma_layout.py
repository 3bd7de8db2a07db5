"""Inner scales in the tensor-core (128 x 4 tiled) layout: every kernel path
writes the oracle's scales in the oracle's statement of the layout (padding
zero), codes unchanged; dequantize reads the layout; and NVFP4 GEMMs in torch
(cuBLASLt) consume the codes and scales of to_fp4_operands as written."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import host_np, oracle_quantize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


@pytest.fixture(params=["fast", "ctb", "tile", "general"])
def kernel(request, monkeypatch):
    for v in ("FP4Q_GENERAL_KERNEL", "FP4Q_NO_ROW_KERNEL", "FP4Q_NO_CTB_KERNEL", "FP4Q_NO_CTL_KERNEL"):
        monkeypatch.delenv(v, raising=False)
    if request.param == "ctb":
        monkeypatch.setenv("FP4Q_NO_CTL_KERNEL", "1")
    elif request.param == "general":
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
def test_mma_layout_equals_oracle(orc, case, shape, dtype, kernel):
    G, M, K = shape
    ob = case.get("outer_block_size", 0)
    if ob and (K % ob or M % ob):
        pytest.skip("shape not divisible by the outer block")
    xc = W.lognormal(shape, 61, sigma=3.0, dtype=dtype)
    x = xc.cuda()
    for mask in ((True, False), (False, True), (True, True)):
        kw = dict(case, rowwise=mask[0], columnwise=mask[1])
        lin = fq.quantize(x, **kw)
        mma = fq.quantize(x, scale_layout="mma", **kw)
        ref = oracle_quantize(orc, xc, **kw)
        for o in ("row", "col"):
            if getattr(lin, o + "_codes") is None:
                continue
            assert (host_np(getattr(mma, o + "_codes")) == ref[o + "_codes"]).all(), (o, kw)
            want = orc.scale_layout_mma(ref[o + "_scales"])
            got = host_np(getattr(mma, o + "_scales"))
            assert got.shape == want.shape and (got == want).all(), (o, kw)
            y_lin = fq.dequantize(lin, o, torch.float32)
            y_mma = fq.dequantize(mma, o, torch.float32)
            assert torch.equal(y_lin.view(torch.int32), y_mma.view(torch.int32))


def test_mma_layout_padding_is_zero_on_reused_buffers(orc):
    """Padding bytes are cleared by every call, also in a reused buffer."""
    xc = W.lognormal((1, 208, 336), 62, sigma=2.0)
    x = xc.cuda()
    q = fq.quantize(x, scale_layout="mma", rowwise=True, columnwise=True)
    q.row_scales.fill_(0xAB)
    q.col_scales.fill_(0xCD)
    fq.quantize(x, scale_layout="mma", rowwise=True, columnwise=True, out=q)
    ref = oracle_quantize(orc, xc, rowwise=True, columnwise=True)
    assert (host_np(q.row_scales) == orc.scale_layout_mma(ref["row_scales"])).all()
    assert (host_np(q.col_scales) == orc.scale_layout_mma(ref["col_scales"])).all()


def _scaled_mm_nvfp4(a, b):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no float4_e2m1fn_x2")
    try:
        return torch._scaled_mm(a.codes, b.codes.t(), a.scales, b.scales, out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip("torch._scaled_mm has no NVFP4 path here: %s" % str(e).splitlines()[0][:120])


def test_to_fp4_operands_types_and_bytes(orc):
    """fp4-train README, "API": to_fp4_operands returns the packed codes and
    the E4M3 scales as torch's FP4 / FP8 dtypes, scales in the tensor-core
    layout; their bytes are the oracle's."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no float4_e2m1fn_x2")
    xc = W.lognormal((208, 320), 65, sigma=2.0)
    for stochastic in (False, True):
        op = fq.to_fp4_operands(xc.cuda(), stochastic=stochastic, seed=4, step=7)
        assert op.codes.dtype == torch.float4_e2m1fn_x2 and tuple(op.codes.shape) == (208, 160)
        assert op.scales.dtype == torch.float8_e4m3fn
        ref = oracle_quantize(orc, xc, stochastic=stochastic, seed=4, step=7)
        assert (host_np(op.codes.view(torch.uint8)) == ref["row_codes"][0]).all()
        assert (host_np(op.scales.view(torch.uint8)) == orc.scale_layout_mma(ref["row_scales"])).all()


@pytest.mark.parametrize("mnk", [(256, 384, 512), (208, 128, 320)], ids=["aligned", "padded"])
def test_nvfp4_gemm_reads_the_layout(mnk):
    """A block-scaled FP4 GEMM (cuBLASLt through torch) reads the operands of
    to_fp4_operands: its result equals the product of the dequantized
    operands up to binary32 accumulation order and the bf16 output rounding.
    A misplaced scale would change results by factors of 2 or more."""
    M, N, K = mnk
    a = W.lognormal((M, K), 63, sigma=2.0).cuda()
    b = W.lognormal((N, K), 64, sigma=2.0).cuda()
    oa, ob_ = fq.to_fp4_operands(a), fq.to_fp4_operands(b)
    y = _scaled_mm_nvfp4(oa, ob_)
    da = fq.dequantize(oa.quantized, "row", torch.float32)[0].double()
    db = fq.dequantize(ob_.quantized, "row", torch.float32)[0].double()
    ref = da @ db.t()
    err = (y.double() - ref).abs()
    tol = 1e-2 * (da.abs() @ db.abs().t()) + 1e-30
    assert (err <= tol).all(), float((err / tol).max())
