"""Tensors past 2^31 elements: the 64-bit index paths of the cast-transpose
and dequantize kernels (the flat MXFP4 and rowwise kernels are covered by
test_gpu_parity.py's test_beyond_2p31_elements).  A bf16 [262272, 8192]
tensor (2^31 + 2^20 elements, 4.3 GB; element 2^31 starts row 262144) is
processed whole, and rows on both sides of element 2^31, the first and the
last rows, and a 128-row slab across it are compared with the oracle bit
for bit.  The oracle takes them as tensors of their own: each method here is
independent per row, or per 16- and 64-row column block, and the slab starts
on a 64-row boundary.  The columnwise index k M + m passes 2^31 in the
slab's last columns."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import assert_same, host_np, oracle_quantize

pytestmark = pytest.mark.gpu

M, K = 262144 + 128, 8192
ROWS = [0, 1, 262143, 262144, 262145, M - 2, M - 1]
S0, S1 = 262144 - 64, 262144 + 64  # the slab across element 2^31
OB = 64


@pytest.fixture(scope="module")
def x():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    if torch.cuda.mem_get_info()[0] < (24 << 30):
        pytest.skip("needs about 16 GB of free device memory")
    t = W.large_rows(M, K, seed=91)
    yield t
    del t
    torch.cuda.empty_cache()


def _rows(t, rows):
    return t[rows].cpu()


def test_rowwise_outer_block_and_dequantize_past_2_31(orc, x):
    kw = dict(mode="outer_block", outer_block_size=OB)
    q = fq.quantize(x, **kw)  # rowwise only: the flat rowwise kernel
    torch.cuda.synchronize()
    ref = oracle_quantize(orc, _rows(x, ROWS), **kw)
    got = {k: host_np(getattr(q, k)[0][ROWS]) for k in ("row_codes", "row_scales", "row_outer")}
    assert_same(got, ref)
    y = fq.dequantize(q)
    torch.cuda.synchronize()
    yref = orc.dequantize(ref["row_codes"], ref["row_scales"], {"row_outer": ref["row_outer"]},
                          G=1, M=len(ROWS), K=K, mode="outer_block", ob=OB)
    assert np.array_equal(host_np(y[0][ROWS]), yref[0])
    del q, y


def test_cast_transpose_past_2_31(orc, x):
    kw = dict(mode="outer_block", outer_block_size=OB, rowwise=True, columnwise=True)
    q = fq.quantize(x, **kw)
    torch.cuda.synchronize()
    ref = oracle_quantize(orc, x[S0:S1].cpu(), **kw)
    got = {
        "row_codes": host_np(q.row_codes[0][S0:S1]),
        "row_scales": host_np(q.row_scales[0][S0:S1]),
        "row_outer": host_np(q.row_outer[0][S0:S1]),
        "col_codes": host_np(q.col_codes[0][:, S0 // 2:S1 // 2]),
        "col_scales": host_np(q.col_scales[0][:, S0 // 16:S1 // 16]),
        "col_outer": host_np(q.col_outer[0][:, S0 // OB:S1 // OB]),
    }
    assert_same(got, ref)
    # the first and last rows too
    for r0 in (0, M - 128):
        ref = oracle_quantize(orc, x[r0:r0 + 128].cpu(), **kw)
        got = {"row_codes": host_np(q.row_codes[0][r0:r0 + 128]),
               "col_codes": host_np(q.col_codes[0][:, r0 // 2:(r0 + 128) // 2]),
               "col_outer": host_np(q.col_outer[0][:, r0 // OB:(r0 + 128) // OB])}
        assert_same(got, ref, keys=list(got))
    del q
