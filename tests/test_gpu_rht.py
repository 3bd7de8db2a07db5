"""Columnwise quantization after the random Hadamard transform along M
against the oracle, bit for bit: modes none and 1-D outer blocks, both masks,
RNE and SR, several sign masks, special values and a block whose sums
overflow binary32, ragged tiles and the tensor-core scale layout."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

from gpu_helpers import assert_same, gpu_quantize, oracle_kw, host_np, to_mma_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


def _oracle(orc, x, kw):
    m = (1 if kw.get("rowwise", True) else 0) | (2 if kw.get("columnwise", False) else 0)
    xo = host_np(x)
    return orc.quantize(xo if xo.ndim == 3 else xo[None], out_mask=m, col_hadamard=True,
                        hadamard_signs=kw["hadamard_signs"], **oracle_kw(kw))


CASES = [dict(mode="none"), dict(mode="outer_block", outer_block_size=16), dict(mode="outer_block", outer_block_size=32),
         dict(mode="outer_block", outer_block_size=64, scale_format="ue5m3"), dict(mode="none", stochastic=True, seed=5)]


@pytest.mark.parametrize("signs", [0, 0xFFFF, 0xA5C3])
@pytest.mark.parametrize("case", CASES, ids=["none", "ob16", "ob32", "ob64-ue5m3", "sr"])
def test_rht_matches_oracle(orc, case, signs):
    x = W.lognormal((1, 192, 320), 91, sigma=2.5)
    x.view(-1)[37] = float("nan")
    x.view(-1)[5000] = float("-inf")
    x[0, 64:80, 17] = 3.3895314e38  # a column block whose butterfly sums overflow
    for mask in ((False, True), (True, True)):
        kw = dict(case, rowwise=mask[0], columnwise=mask[1], col_hadamard=True, hadamard_signs=signs)
        _, g = gpu_quantize(x, **kw)
        r = _oracle(orc, x, kw)
        assert_same(g, r)



@pytest.mark.parametrize("case", [dict(mode="none"), dict(mode="outer_block", outer_block_size=64),
                                  dict(mode="outer_block", outer_block_size=64, scale_format="ue5m3")],
                         ids=["none", "ob64", "ob64-ue5m3"])
def test_rht_whole_tiles(orc, case):
    """M a multiple of 128 and K of 64: the kernel's whole-tile form, with a
    block whose butterfly sums overflow, a zero 64-row column group and a
    block of tiny values (the general per-block steps)."""
    x = W.lognormal((2, 256, 192), 93, sigma=2.5)
    x[1, 128:144, 70] = 3.3895314e38
    x[0, 0:64, 5] = 0.0
    x[0, 128:144, 9] *= 1e-30
    for mask in ((False, True), (True, True)):
        kw = dict(case, rowwise=mask[0], columnwise=mask[1], col_hadamard=True, hadamard_signs=0x5A0F)
        _, g = gpu_quantize(x, **kw)
        assert_same(g, _oracle(orc, x, kw))

def test_rht_all_bf16_patterns_and_mma_layout(orc):
    x = W.all_bf16_patterns()
    kw = dict(mode="outer_block", outer_block_size=32, rowwise=True, columnwise=True, col_hadamard=True,
              hadamard_signs=0x1234)
    q, g = gpu_quantize(x, **kw)
    r = _oracle(orc, x, kw)
    assert_same(g, r)
    qm = fq.quantize(x.cuda(), scale_layout="mma", **kw)
    assert torch.equal(qm.col_codes, q.col_codes)
    assert (host_np(qm.col_scales) == to_mma_layout(host_np(q.col_scales))).all()


def test_rht_rejections():
    x = W.lognormal((1, 64, 64), 92).cuda()
    with pytest.raises(fq.FP4QError):
        fq.quantize(x, columnwise=True, mode="tensorwise", col_hadamard=True)
    with pytest.raises(fq.FP4QError):
        fq.quantize(x, columnwise=True, mode="outer_block", outer_block_size=64, outer_2d=True, col_hadamard=True)
    with pytest.raises(fq.FP4QError):
        fq.quantize(x.float(), columnwise=True, col_hadamard=True)
    with pytest.raises(fq.FP4QError):
        fq.quantize(x, rowwise=True, columnwise=False, col_hadamard=True)
