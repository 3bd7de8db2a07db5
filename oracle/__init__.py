"""CPU oracle for the block-scaled FP4 quantizer.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain statement of what
the quantizer computes (scalar C99 in ``fp4_oracle.c``, binary32 arithmetic,
no FMA contraction, subnormals kept).  Only the test-suite, the smoke check
and the CPU-baseline leg of ``bench.py`` may import it; the library's product
path never does, and the two share no code.

Arrays are numpy.  bfloat16 data is carried as ``np.uint16`` bit patterns,
binary32 as ``np.float32``.  Shapes follow the library's layout:

* input ``x``: ``[G, M, ld]`` (``ld >= K``; pass ``K`` when ``ld > K``)
* rowwise codes ``[G, M, K/2]`` (two E2M1 codes per byte, even column in the
  low nibble), inner scales ``[G, M, K/16]``
* columnwise codes ``[G, K, M/2]``, inner scales ``[G, K, M/16]``
* outer scales: 1-D rowwise ``[G, M, K/ob]``, 1-D columnwise ``[G, K, M/ob]``,
  2-D ``[G, M/ob, K/ob]`` (shared), tensorwise ``[1]``

* inner scales in the tensor-core layout (``scale_layout_mma``): flat bytes,
  128 x 4 blocks of 512 bytes per matrix

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
except the Philox stream beyond its published known-answer vectors and the
statistics of stochastic rounding ("parity unpinned" for the exact SR word
assignment, which is this library's own definition).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4_oracle.c")
_SO = os.path.join(_HERE, "_build", "liborc.so")

BF16, FP32 = 1, 2
MODE_NONE, MODE_TENSORWISE, MODE_OUTER = 0, 1, 2
E4M3, UE5M3 = 0, 1
RNE, SR = 0, 1
ROW, COL = 1, 2

_MODES = {"none": MODE_NONE, "tensorwise": MODE_TENSORWISE, "outer_block": MODE_OUTER}
_FMTS = {"e4m3": E4M3, "ue5m3": UE5M3}


def build(force: bool = False) -> str:
    """Compile the oracle into a shared object next to this file."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class Cfg(ctypes.Structure):
    _fields_ = [
        ("G", ctypes.c_int64), ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("ld", ctypes.c_int64),
        ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("mode", ctypes.c_int32),
        ("ob", ctypes.c_int32), ("outer_2d", ctypes.c_int32), ("inner_2d", ctypes.c_int32),
        ("fmt", ctypes.c_int32), ("rounding", ctypes.c_int32), ("seed", ctypes.c_uint64),
        ("step", ctypes.c_uint32), ("out_mask", ctypes.c_uint32), ("use_precomputed", ctypes.c_int32),
        ("sr_index_base", ctypes.c_int64),
        ("col_hadamard", ctypes.c_int32), ("hadamard_signs", ctypes.c_uint32),
    ]


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_rne.restype = ctypes.c_uint8
        L.orc_e2m1_rne.argtypes = [ctypes.c_double]
        L.orc_e2m1_sr.restype = ctypes.c_uint8
        L.orc_e2m1_sr.argtypes = [ctypes.c_double, ctypes.c_uint32]
        L.orc_scale_decode.restype = ctypes.c_double
        L.orc_scale_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
        L.orc_scale_encode.restype = ctypes.c_uint8
        L.orc_scale_encode.argtypes = [ctypes.c_int, ctypes.c_float]
        L.orc_philox4x32_10.restype = None
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_sr_word.restype = ctypes.c_uint32
        L.orc_sr_word.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64]
        L.orc_mxfp4_exponent.restype = ctypes.c_int
        L.orc_mxfp4_exponent.argtypes = [ctypes.c_double]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_quantize.argtypes = [ctypes.POINTER(Cfg), P, P, P, P, P, P, P, P, P]
        L.orc_dequantize.restype = ctypes.c_int
        L.orc_dequantize.argtypes = [ctypes.POINTER(Cfg), ctypes.c_int, P, P, P, P, P, P]
        L.orc_qdq.restype = ctypes.c_int
        L.orc_qdq.argtypes = [ctypes.POINTER(Cfg), ctypes.c_int, P, P, P, P, P, P]
        L.orc_mxfp4_fake_quantize.restype = ctypes.c_int
        L.orc_mxfp4_fake_quantize.argtypes = [ctypes.POINTER(Cfg), P, P]
        L.orc_mxfp8_exponent.restype = ctypes.c_int
        L.orc_mxfp8_exponent.argtypes = [ctypes.c_double]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_mxfp4_project_mxfp8.restype = ctypes.c_int
        L.orc_mxfp4_project_mxfp8.argtypes = [ctypes.POINTER(Cfg), P, P, P, P, P, P]
        L.orc_rht16.restype = None
        L.orc_rht16.argtypes = [P, ctypes.c_uint32, ctypes.c_int32]
        L.orc_scale_layout_mma.restype = None
        L.orc_scale_layout_mma.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P]
        L.orc_subnormals_ok.restype = ctypes.c_int
        _lib_handle = L
    return _lib_handle


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(arr):
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return FP32
    raise TypeError("oracle input must be uint16 (bf16 bits) or float32, got %s" % arr.dtype)


def _out_np(code):
    return np.uint16 if code == BF16 else np.float32


def _as3d(x):
    x = np.ascontiguousarray(x)
    if x.ndim == 2:
        x = x[None]
    assert x.ndim == 3
    return x


def make_cfg(x, K=None, *, mode="none", ob=0, outer_2d=False, inner_2d=False, fmt="e4m3",
             rounding="rne", seed=0, step=0, out_mask=ROW, use_precomputed=False, out_dtype=None,
             sr_index_base=0, col_hadamard=False, hadamard_signs=0):
    G, M, ld = x.shape
    K = ld if K is None else K
    in_code = _dtype_code(x)
    out_code = in_code if out_dtype is None else {"bf16": BF16, "fp32": FP32}[out_dtype]
    return Cfg(G, M, K, ld, in_code, out_code, _MODES[mode] if isinstance(mode, str) else mode, ob,
               int(outer_2d), int(inner_2d), _FMTS[fmt] if isinstance(fmt, str) else fmt,
               {"rne": RNE, "sr": SR}[rounding] if isinstance(rounding, str) else rounding,
               seed, step, out_mask, int(use_precomputed), int(sr_index_base), int(bool(col_hadamard)),
               int(hadamard_signs) & 0xFFFFFFFF)


def outer_shapes(cfg):
    G, M, K, ob = cfg.G, cfg.M, cfg.K, cfg.ob
    shapes = {"row_outer": None, "col_outer": None, "tile_outer": None}
    if cfg.mode == MODE_TENSORWISE:
        shapes["tile_outer"] = (1,)
    elif cfg.mode == MODE_OUTER:
        if cfg.outer_2d:
            shapes["tile_outer"] = (G, M // ob, K // ob)
        else:
            if cfg.out_mask & ROW:
                shapes["row_outer"] = (G, M, K // ob)
            if cfg.out_mask & COL:
                shapes["col_outer"] = (G, K, M // ob)
    return shapes


def _outer_bufs(cfg, precomputed):
    bufs = {}
    for name, shp in outer_shapes(cfg).items():
        if shp is None:
            bufs[name] = None
        elif precomputed is not None and precomputed.get(name) is not None:
            bufs[name] = np.ascontiguousarray(precomputed[name], dtype=np.float32).reshape(shp).copy()
        else:
            bufs[name] = np.zeros(shp, np.float32)
    return bufs


def quantize(x, K=None, *, residual=None, precomputed=None, **kw):
    """Quantize ``x`` ([G,M,ld] or [M,ld]); returns a dict of numpy outputs.

    ``residual`` ([G,M,K] float32, rowwise only) is updated in place.
    ``precomputed`` (dict of outer-scale arrays) is read when
    ``use_precomputed=True``."""
    x = _as3d(x)
    cfg = make_cfg(x, K, **kw)
    G, M, Kk = cfg.G, cfg.M, cfg.K
    out = {}
    if cfg.out_mask & ROW:
        out["row_codes"] = np.zeros((G, M, Kk // 2), np.uint8)
        out["row_scales"] = np.zeros((G, M, Kk // 16), np.uint8)
    if cfg.out_mask & COL:
        out["col_codes"] = np.zeros((G, Kk, M // 2), np.uint8)
        out["col_scales"] = np.zeros((G, Kk, M // 16), np.uint8)
    out.update(_outer_bufs(cfg, precomputed if cfg.use_precomputed else None))
    if residual is not None:
        assert residual.dtype == np.float32 and residual.flags.c_contiguous and residual.size == G * M * Kk
    rc = _lib().orc_quantize(ctypes.byref(cfg), _ptr(x), _ptr(residual),
                             _ptr(out.get("row_codes")), _ptr(out.get("row_scales")), _ptr(out["row_outer"]),
                             _ptr(out.get("col_codes")), _ptr(out.get("col_scales")), _ptr(out["col_outer"]),
                             _ptr(out["tile_outer"]))
    assert rc == 0
    return out


def dequantize(codes, scales, outer, *, G, M, K, orient=ROW, out_dtype="bf16", mode="none", ob=0,
               outer_2d=False, fmt="e4m3"):
    """Dequantize one orientation's buffers; returns [G,R,C] in ``out_dtype``."""
    dummy = np.zeros((G, M, K), np.float32)
    cfg = make_cfg(dummy, None, mode=mode, ob=ob, outer_2d=outer_2d, fmt=fmt, out_mask=orient,
                   out_dtype=out_dtype)
    R, C = (M, K) if orient == ROW else (K, M)
    y = np.zeros((G, R, C), _out_np(cfg.out_dtype))
    outer = outer or {}
    bufs = {k: (None if outer.get(k) is None else np.ascontiguousarray(outer[k], dtype=np.float32))
            for k in ("row_outer", "col_outer", "tile_outer")}
    rc = _lib().orc_dequantize(ctypes.byref(cfg), orient, _ptr(np.ascontiguousarray(codes)),
                               _ptr(np.ascontiguousarray(scales)), _ptr(bufs["row_outer"]),
                               _ptr(bufs["col_outer"]), _ptr(bufs["tile_outer"]), _ptr(y))
    assert rc == 0
    return y


def qdq(x, K=None, *, orient=ROW, residual=None, precomputed=None, **kw):
    """Quantize then dequantize along ``orient`` (ROW: along K, COL: along M).

    Returns (y [G,M,K] in the output dtype, dict of outer scales)."""
    x = _as3d(x)
    kw = dict(kw)
    kw["out_mask"] = orient
    cfg = make_cfg(x, K, **kw)
    y = np.zeros((cfg.G, cfg.M, cfg.K), _out_np(cfg.out_dtype))
    bufs = _outer_bufs(cfg, precomputed if cfg.use_precomputed else None)
    rc = _lib().orc_qdq(ctypes.byref(cfg), orient, _ptr(x), _ptr(y), _ptr(residual),
                        _ptr(bufs["row_outer"]), _ptr(bufs["col_outer"]), _ptr(bufs["tile_outer"]))
    assert rc == 0
    return y, bufs


def mxfp4_fake_quantize(x, K=None, *, out_dtype=None):
    """MXFP4 fake-quantize (1x32 power-of-two scales, RNE); returns [G,M,K]."""
    x = _as3d(x)
    cfg = make_cfg(x, K, out_dtype=out_dtype)
    y = np.zeros((cfg.G, cfg.M, cfg.K), _out_np(cfg.out_dtype))
    rc = _lib().orc_mxfp4_fake_quantize(ctypes.byref(cfg), _ptr(x), _ptr(y))
    assert rc == 0
    return y


def mxfp4_project_mxfp8(x, K=None, *, out_dtype=None, out_mask=ROW | COL, with_y=True):
    """MXFP4 projection and its MXFP8 encodings (OCP MX reading, see the C
    source): returns dict y [G,M,K] (or None), row_codes [G,M,K] u8 (E4M3),
    row_scales [G,M,K/32] u8 (UE8M0), col_codes [G,K,M], col_scales
    [G,K,M/32] for the orientations in out_mask."""
    x = _as3d(x)
    cfg = make_cfg(x, K, out_dtype=out_dtype)
    G, M, Kk = cfg.G, cfg.M, cfg.K
    out = {"y": np.zeros((G, M, Kk), _out_np(cfg.out_dtype)) if with_y else None,
           "row_codes": None, "row_scales": None, "col_codes": None, "col_scales": None}
    if out_mask & ROW:
        out["row_codes"] = np.zeros((G, M, Kk), np.uint8)
        out["row_scales"] = np.zeros((G, M, Kk // 32), np.uint8)
    if out_mask & COL:
        assert M % 32 == 0
        out["col_codes"] = np.zeros((G, Kk, M), np.uint8)
        out["col_scales"] = np.zeros((G, Kk, M // 32), np.uint8)
    rc = _lib().orc_mxfp4_project_mxfp8(ctypes.byref(cfg), _ptr(x), _ptr(out["y"]), _ptr(out["row_codes"]),
                                       _ptr(out["row_scales"]), _ptr(out["col_codes"]), _ptr(out["col_scales"]))
    assert rc == 0
    return out


def scale_layout_mma(lin):
    """An orientation's [G, R, C] (or [R, C]) linear inner-scale bytes in the
    tensor-core layout (128 x 4 blocks of 512 bytes, zero padding); returns
    the flat byte buffer."""
    a = np.ascontiguousarray(lin, np.uint8)
    if a.ndim == 2:
        a = a[None]
    G, R, C = a.shape
    out = np.zeros(G * (-(-R // 128)) * (-(-C // 4)) * 512, np.uint8)
    _lib().orc_scale_layout_mma(_ptr(a), G, R, C, _ptr(out))
    return out


def rht16(v, signs: int, in_dtype: str = "fp32"):
    """The oracle's 16-point random Hadamard transform of one block (float32)."""
    a = np.ascontiguousarray(np.asarray(v, np.float32).copy())
    assert a.shape == (16,)
    _lib().orc_rht16(_ptr(a), int(signs) & 0xFFFFFFFF, BF16 if in_dtype == "bf16" else FP32)
    return a


def mxfp8_exponent(A: float) -> int:
    return _lib().orc_mxfp8_exponent(float(A))


def e4m3_encode(v: float) -> int:
    return _lib().orc_e4m3_encode(float(v))


# ---- scalar helpers (for pins) ------------------------------------------

def e2m1_rne(t: float) -> int:
    return _lib().orc_e2m1_rne(float(t))


def e2m1_sr(t: float, w: int) -> int:
    return _lib().orc_e2m1_sr(float(t), int(w))


def e2m1_decode(code: int) -> float:
    return _lib().orc_e2m1_decode(code)


def scale_encode(fmt, v: float) -> int:
    return _lib().orc_scale_encode(_FMTS.get(fmt, fmt), float(v))


def scale_decode(fmt, c: int) -> float:
    return _lib().orc_scale_decode(_FMTS.get(fmt, fmt), int(c))


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, np.uint32).copy()
    k = np.asarray(key, np.uint32).copy()
    o = np.zeros(4, np.uint32)
    _lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return [int(v) for v in o]


def sr_word(seed: int, step: int, orient: int, n: int) -> int:
    return _lib().orc_sr_word(seed, step, orient, n)


def mxfp4_exponent(A: float) -> int:
    return _lib().orc_mxfp4_exponent(float(A))


def f32_to_bf16(v: float) -> int:
    return _lib().orc_f32_to_bf16(float(v))


def bf16_to_f32(h: int) -> float:
    return _lib().orc_bf16_to_f32(int(h))


def subnormals_ok() -> bool:
    return bool(_lib().orc_subnormals_ok())
