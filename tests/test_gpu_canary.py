"""Guard zones: every output buffer is carved out of a larger allocation
whose head and tail bytes hold a known pattern.  After each entry point the
pattern is intact (no write outside an output) and the outputs equal those
of a call with buffers of their own.  The shapes are ragged (M not a
multiple of the 128-row tile, K not a multiple of the 64-column tile, block
counts that do not fill a warp), so every kernel's edge handling runs:
the flat rowwise kernel, the bf16 and binary32 cast-transpose kernels, the
general tile kernel (16x16 inner blocks), the outer-scale pre-pass, the
tensor-core scale layout, the grouped path, QDQ, dequantize, MXFP4 and the
MXFP4 -> MXFP8 re-encode."""
import dataclasses

import pytest
import torch

import block_scaled_fp4_quantize_gb300 as fq
from block_scaled_fp4_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096        # guard bytes on each side (keeps 256-byte alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()


class Arena:
    """Carves guarded views; check() asserts every guard is intact."""

    def __init__(self):
        self.backs = []

    def like(self, t):
        if t is None:
            return None
        nbytes = t.numel() * t.element_size()
        back = torch.full((2 * GUARD + nbytes,), PATTERN, dtype=torch.uint8, device="cuda")
        self.backs.append((back, nbytes))
        return back[GUARD:GUARD + nbytes].view(t.dtype).view(t.shape)

    def check(self):
        for back, nbytes in self.backs:
            head, tail = back[:GUARD], back[GUARD + nbytes:]
            assert bool((head == PATTERN).all()), "write before an output buffer"
            assert bool((tail == PATTERN).all()), "write past an output buffer"


FIELDS = ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer")


def _guarded_q(q, arena):
    return dataclasses.replace(q, **{f: arena.like(getattr(q, f)) for f in FIELDS})


def _same_q(a, b):
    for f in FIELDS:
        x, y = getattr(a, f), getattr(b, f)
        assert (x is None) == (y is None), f
        if x is not None:
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), f


QUANT_CASES = [
    ("row-flat", (1, 80, 176), torch.bfloat16, dict(mode="outer_block", outer_block_size=16), True, False),
    ("ct-bf16-ob16", (1, 80, 176), torch.bfloat16, dict(mode="outer_block", outer_block_size=16), True, True),
    ("ct-bf16-ob64", (2, 192, 320), torch.bfloat16, dict(mode="outer_block", outer_block_size=64), True, True),
    ("ct-bf16-prepass-ob48", (2, 96, 144), torch.bfloat16, dict(mode="outer_block", outer_block_size=48), True, True),
    ("ct-bf16-2d", (1, 192, 192), torch.bfloat16, dict(mode="outer_block", outer_block_size=64, outer_2d=True),
     True, True),
    ("ct-bf16-tensorwise", (1, 80, 176), torch.bfloat16, dict(mode="tensorwise"), True, True),
    ("ct-bf16-none-ue5m3", (1, 80, 176), torch.bfloat16, dict(mode="none", scale_format="ue5m3"), True, True),
    ("ct-bf16-mma", (1, 80, 176), torch.bfloat16, dict(mode="outer_block", outer_block_size=16, scale_layout="mma"),
     True, True),
    ("ct-bf16-sr", (1, 80, 176), torch.bfloat16, dict(mode="outer_block", outer_block_size=16, stochastic=True,
                                                      seed=5, step=2), True, True),
    ("ct-bf16-hadamard", (1, 80, 176), torch.bfloat16, dict(mode="outer_block", outer_block_size=16,
                                                            col_hadamard=True, hadamard_signs=0x1234), True, True),
    ("ct-fp32", (1, 80, 176), torch.float32, dict(mode="outer_block", outer_block_size=16), True, True),
    # whole tiles (M a multiple of 128, K of 64): the kernels' no-edge forms
    ("ct-bf16-whole-ob64", (2, 256, 192), torch.bfloat16, dict(mode="outer_block", outer_block_size=64), True, True),
    ("ct-bf16-whole-2d", (1, 128, 128), torch.bfloat16, dict(mode="outer_block", outer_block_size=64, outer_2d=True),
     True, True),
    ("ct-bf16-whole-none", (1, 128, 320), torch.bfloat16, dict(mode="none"), True, True),
    ("ct-bf16-whole-tensorwise", (3, 128, 64), torch.bfloat16, dict(mode="tensorwise"), True, True),
    ("tile-inner2d", (1, 96, 96), torch.bfloat16, dict(mode="outer_block", outer_block_size=32, inner_2d=True),
     True, True),
]


@pytest.mark.parametrize("name,shape,dtype,kw,row,col", QUANT_CASES, ids=[c[0] for c in QUANT_CASES])
def test_quantize_writes_only_its_outputs(name, shape, dtype, kw, row, col):
    x = W.lognormal(shape, 71, sigma=3.0, dtype=dtype).cuda()
    ref = fq.quantize(x, rowwise=row, columnwise=col, **kw)
    arena = Arena()
    q = _guarded_q(ref, arena)
    got = fq.quantize(x, rowwise=row, columnwise=col, out=q, **kw)
    torch.cuda.synchronize()
    arena.check()
    _same_q(got, ref)
    # dequantize each orientation into a guarded output
    if not kw.get("inner_2d") and kw.get("scale_layout", "linear") == "linear":
        for orient in (["row"] if row else []) + (["col"] if col else []):
            y0 = fq.dequantize(ref, orient)
            y = arena.like(y0)
            fq.dequantize(got, orient, out=y)
            torch.cuda.synchronize()
            arena.check()
            assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("axis", [-1, 0])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_qdq_writes_only_its_output(axis, dtype):
    x = W.lognormal((1, 80, 176), 72, sigma=3.0, dtype=dtype).cuda()
    kw = dict(mode="outer_block", outer_block_size=16)
    y0, _ = fq.qdq(x, axis=axis, **kw)
    arena = Arena()
    y = arena.like(y0)
    fq.qdq(x, axis=axis, out=y, **kw)
    torch.cuda.synchronize()
    arena.check()
    assert torch.equal(y.view(torch.uint8), y0.view(torch.uint8))


def test_grouped_quantize_writes_only_its_outputs():
    x = W.lognormal((1, 320, 192), 73, sigma=2.0)[0].cuda()
    off = torch.tensor([0, 64, 64, 256, 320], dtype=torch.int64, device="cuda")
    kw = dict(mode="outer_block", outer_block_size=64, rowwise=True, columnwise=True)
    ref = fq.quantize_grouped(x, off, **kw)
    arena = Arena()
    q = _guarded_q(ref, arena)
    got = fq.quantize_grouped(x, off, out=q, **kw)
    torch.cuda.synchronize()
    arena.check()
    _same_q(got, ref)


@pytest.mark.parametrize("shape", [(1, 100, 96), (3, 7, 64)], ids=["100x96", "3x7x64"])
def test_mxfp4_writes_only_its_output(shape):
    x = W.lognormal(shape, 74, sigma=6.0).cuda()
    y0 = fq.mxfp4_fake_quantize(x)
    arena = Arena()
    y = arena.like(y0)
    fq.mxfp4_fake_quantize(x, out=y)
    torch.cuda.synchronize()
    arena.check()
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


def test_mxfp8_writes_only_its_outputs():
    x = W.lognormal((1, 160, 96), 75, sigma=4.0).cuda()
    ref = fq.mxfp4_project_mxfp8(x, with_y=True)
    arena = Arena()
    out = fq.MXFP8Pair(**{f.name: arena.like(getattr(ref, f.name)) for f in dataclasses.fields(ref)})
    got = fq.mxfp4_project_mxfp8(x, with_y=True, out=out)
    torch.cuda.synchronize()
    arena.check()
    for f in dataclasses.fields(ref):
        assert torch.equal(getattr(got, f.name).view(torch.uint8), getattr(ref, f.name).view(torch.uint8)), f.name
