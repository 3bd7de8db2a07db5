"""Host-side tests of the C ABI: the library loads, exports every symbol the
header declares, and its argument validation returns the documented codes.

Every call here fails validation before the library touches CUDA, so the
tests run without a GPU.  (Pointers passed are never dereferenced.)
"""
import ctypes
import os
import re

import pytest

from block_scaled_fp4_quantize_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4q.h")

FAKE = ctypes.c_void_p(0x100000)  # 256-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    return _capi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;]*\)\s*;", text, re.M))


def test_header_declares_the_bound_functions():
    assert declared_functions() == set(_capi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.fp4q_abi_version() == 4
    out = os.popen("nm -D --defined-only %s" % _capi._build.lib_path()).read()
    for name in declared_functions():
        assert re.search(r"\sT\s%s$" % name, out, re.M), name


def test_params_struct_layout_matches(lib):
    p = _capi.Params()
    lib.fp4q_params_init(ctypes.byref(p))
    assert p.struct_size == ctypes.sizeof(_capi.Params) == 128
    assert (p.G, p.in_dtype, p.out_dtype, p.mode, p.out_mask, p.scale_layout) == (1, _capi.BF16, _capi.BF16, 0, 1, 0)
    assert (p.precomputed_amax, p.sr_global_rows, p.sr_row_offset, p.sr_matrix_offset) == (0, 0, 0, 0)
    assert ctypes.sizeof(_capi.Outputs) == 7 * 8 and ctypes.sizeof(_capi.Sizes) == 8 * 8


def mk(lib, **kw):
    p = _capi.new_params(lib)
    p.M, p.K, p.ld = 128, 256, 256
    for k, v in kw.items():
        setattr(p, k, v)
    if "ld" not in kw:
        p.ld = p.K
    return p


def sizes(lib, **kw):
    s = _capi.Sizes()
    rc = lib.fp4q_query_sizes(ctypes.byref(mk(lib, **kw)), ctypes.byref(s))
    return rc, s


def test_query_sizes(lib):
    rc, s = sizes(lib, G=2, M=128, K=256, mode=2, outer_block_size=64, out_mask=3)
    assert rc == 0
    assert (s.row_codes, s.row_scales, s.col_codes, s.col_scales) == (2 * 128 * 128, 2 * 128 * 16, 2 * 256 * 64,
                                                                      2 * 256 * 8)
    assert (s.row_outer, s.col_outer, s.tile_outer, s.workspace) == (2 * 128 * 4 * 4, 2 * 256 * 2 * 4, 0, 0)
    rc, s = sizes(lib, M=128, K=256, mode=2, outer_block_size=64, outer_2d=1, out_mask=3)
    assert rc == 0 and (s.row_outer, s.col_outer, s.tile_outer) == (0, 0, 2 * 4 * 4)
    rc, s = sizes(lib, mode=1)
    assert rc == 0 and s.tile_outer == 4 and s.workspace == 256
    rc, s = sizes(lib, mode=1, use_precomputed_outer=1)
    assert rc == 0 and s.workspace == 0


@pytest.mark.parametrize("kw,code", [
    (dict(in_dtype=_capi.FP16), -2),                       # fp16 rejected (MXFP4 QAT page, "Guards")
    (dict(in_dtype=7), -2),
    (dict(K=72, ld=72), -3),                               # K % 16
    (dict(ld=100), -3),                                    # ld < K
    (dict(M=40, out_mask=3), -3),                          # M % 16 with columnwise
    (dict(M=40, inner_2d=1), -3),                          # M % 16 with 16x16 inner blocks
    (dict(mode=2, outer_block_size=24), -3),               # ob % 16
    (dict(mode=2, outer_block_size=96), -3),               # ob does not divide K = 256
    (dict(mode=2, outer_block_size=64, M=96, outer_2d=1), -3),  # ob does not divide M (2-D)
    (dict(mode=2, outer_block_size=0), -3),
    (dict(mode=1, outer_block_size=64), -4),               # outer knobs outside outer-block mode
    (dict(mode=0, outer_2d=1), -4),
    (dict(mode=0, use_precomputed_outer=1), -4),
    (dict(mode=5), -4),
    (dict(out_mask=0), -4),
    (dict(out_mask=4), -4),
    (dict(scale_format=3), -4),
    (dict(rounding=2), -4),
    (dict(struct_size=80), -8),
    (dict(struct_size=104), -8),                           # the previous ABI's struct
    (dict(precomputed_amax=1), -4),                        # precomputed amax outside tensorwise mode
    (dict(mode=1, precomputed_amax=1, use_precomputed_outer=1), -4),
    (dict(mode=1, precomputed_amax=2), -4),
    (dict(sr_global_rows=-1), -3),                         # SR counter's global index
    (dict(sr_global_rows=200, sr_row_offset=100), -3),     # rows 100 .. 228 of 200
    (dict(sr_row_offset=4), -3),                           # an offset needs the global row count
    (dict(sr_matrix_offset=-2), -3),
    (dict(G=2, sr_global_rows=512), -5),                   # several matrices must be whole
])
def test_validation_codes(lib, kw, code):
    rc, _ = sizes(lib, **kw)
    assert rc == code
    out = _capi.Outputs(*([FAKE] * 7))
    assert lib.fp4_quantize(ctypes.byref(mk(lib, **kw)), FAKE, ctypes.byref(out), None, FAKE, 256, None) == code


def test_quantize_guards(lib):
    out = _capi.Outputs(*([FAKE] * 7))
    p = mk(lib, out_mask=3)
    # error feedback is defined for the rowwise orientation only
    assert lib.fp4_quantize(ctypes.byref(p), FAKE, ctypes.byref(out), FAKE, None, 0, None) == -5
    # tensorwise needs its workspace
    p = mk(lib, mode=1)
    assert lib.fp4_quantize(ctypes.byref(p), FAKE, ctypes.byref(out), None, None, 0, None) == -6
    assert lib.fp4_quantize(ctypes.byref(p), FAKE, ctypes.byref(out), None, FAKE, 16, None) == -6
    # missing buffers
    p = mk(lib)
    assert lib.fp4_quantize(ctypes.byref(p), None, ctypes.byref(out), None, None, 0, None) == -1
    nocodes = _capi.Outputs(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.fp4_quantize(ctypes.byref(p), FAKE, ctypes.byref(nocodes), None, None, 0, None) == -1
    assert lib.fp4_quantize(None, FAKE, ctypes.byref(out), None, None, 0, None) == -1
    # misaligned code buffer
    bad = _capi.Outputs(ctypes.c_void_p(0x100004), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.fp4_quantize(ctypes.byref(p), FAKE, ctypes.byref(bad), None, None, 0, None) == -9
    # misaligned bf16 input element
    assert lib.fp4_quantize(ctypes.byref(p), ctypes.c_void_p(0x100001), ctypes.byref(out), None, None, 0,
                            None) == -9


def test_qdq_dequant_mxfp4_guards(lib):
    p = mk(lib)
    assert lib.fp4_qdq(ctypes.byref(p), 3, FAKE, FAKE, None, None, None, 0, None) == -4
    assert lib.fp4_qdq(ctypes.byref(p), 2, FAKE, FAKE, FAKE, None, None, 0, None) == -5
    p = mk(lib, mode=2, outer_block_size=64)
    assert lib.fp4_qdq(ctypes.byref(p), 1, FAKE, FAKE, None, None, None, 0, None) == -1  # outer buffer
    p = mk(lib, out_dtype=_capi.FP16)
    assert lib.fp4_qdq(ctypes.byref(p), 1, FAKE, FAKE, None, None, None, 0, None) == -2
    assert lib.fp4_dequantize(ctypes.byref(p), 1, FAKE, FAKE, None, FAKE, None) == -2
    p = mk(lib, mode=1)
    assert lib.fp4_dequantize(ctypes.byref(p), 1, FAKE, FAKE, None, FAKE, None) == -1
    assert lib.fp4_dequantize(ctypes.byref(p), 0, FAKE, FAKE, FAKE, FAKE, None) == -4
    # MXFP4: K % 32, defaults only, RNE only
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib, K=48)), FAKE, FAKE, None) == -3
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib, mode=1)), FAKE, FAKE, None) == -4
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib, scale_format=1)), FAKE, FAKE, None) == -4
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib, rounding=1)), FAKE, FAKE, None) == -5
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib, in_dtype=_capi.FP16)), FAKE, FAKE, None) == -2
    assert lib.mxfp4_fake_quantize(ctypes.byref(mk(lib)), None, FAKE, None) == -1


def test_empty_inputs_enqueue_nothing(lib):
    # zero-sized tensors are valid and return before any CUDA call
    for kw in (dict(M=0), dict(G=0), dict(K=0, ld=0)):
        p = mk(lib, **kw)
        out = _capi.Outputs()
        assert lib.fp4_quantize(ctypes.byref(p), None, ctypes.byref(out), None, None, 0, None) == 0
        assert lib.mxfp4_fake_quantize(ctypes.byref(p), None, None, None) == 0
        assert lib.fp4_dequantize(ctypes.byref(p), 1, None, None, None, None, None) == 0


def test_status_strings(lib):
    for code, name in _capi.STATUS.items():
        assert lib.fp4q_status_string(code).decode().startswith(name)


def test_mma_scale_layout_sizes_and_validation(lib):
    """Tensor-core scale layout: rows padded to 128 and scales per row to 4,
    512-byte tiles per matrix; other layout codes are rejected."""
    for G, M, K in ((1, 208, 336), (3, 128, 256), (2, 16, 64), (1, 4096, 7168)):
        p = mk(lib, G=G, M=M, K=K, out_mask=3, scale_layout=1)
        s = _capi.Sizes()
        assert lib.fp4q_query_sizes(ctypes.byref(p), ctypes.byref(s)) == 0
        cdiv = lambda a, b: -(-a // b)
        assert s.row_scales == G * cdiv(M, 128) * cdiv(K // 16, 4) * 512
        assert s.col_scales == G * cdiv(K, 128) * cdiv(M // 16, 4) * 512
        assert s.row_codes == G * M * K // 2
        p.scale_layout = 0
        assert lib.fp4q_query_sizes(ctypes.byref(p), ctypes.byref(s)) == 0
        assert s.row_scales == G * M * K // 16 and s.col_scales == G * K * M // 16
    p = mk(lib, scale_layout=2)
    assert lib.fp4q_query_sizes(ctypes.byref(p), ctypes.byref(_capi.Sizes())) == -4  # FP4Q_ERR_MODE
    p = mk(lib, scale_layout=1)
    assert lib.mxfp4_fake_quantize(ctypes.byref(p), None, None, None) == -4  # FP4Q_ERR_MODE
