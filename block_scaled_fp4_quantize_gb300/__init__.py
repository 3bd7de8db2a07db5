"""Block-scaled FP4 quantizer for GB300 (sm_103a): NVFP4, AMD-FP4 and MXFP4.

Thin PyTorch binding over the C ABI of ``include/fp4q.h``: torch provides
device memory and the current stream, every step of the computation runs in
the library's CUDA kernels.  The library must be built for the GPU in use
(``build()``); there is no CPU fallback.

    quantize(x, ...)            -> QuantizedFP4 (rowwise / columnwise codes and scales)
    dequantize(q, orient="row") -> bf16 / fp32 tensor
    qdq(x, ...)                 -> (y, outer scales)
    mxfp4_fake_quantize(x)      -> projected tensor
    mxfp4_fake_quantize_host(x) -> the same for a host tensor, streamed through the GPU
    tensor_amax(x)              -> max |x| (sanitized) as a 1-element fp32 tensor
    to_fp4_operands(x)          -> codes / scales as torch FP4 / FP8 tensors for _scaled_mm
    device_status()             -> raises if a kernel's bounded wait ran out
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _capi
from ._capi import FP4QError

__all__ = ["QuantizedFP4", "MXFP8Pair", "quantize", "quantize_grouped", "dequantize", "mxfp4_project_mxfp8", "qdq", "mxfp4_fake_quantize", "mxfp4_fake_quantize_host",
           "tensor_amax", "build", "FP4QError", "query_sizes", "host_workspace_bytes", "tensorwise_workspace",
           "workspace_amax", "device_status", "FP4Operands", "to_fp4_operands"]

_MODES = {"none": _capi.MODE_NONE, "tensorwise": _capi.MODE_TENSORWISE, "outer_block": _capi.MODE_OUTER_BLOCK}
_FMTS = {"e4m3": _capi.SCALE_E4M3, "ue5m3": _capi.SCALE_UE5M3}
_LAYOUTS = {"linear": _capi.SCALE_LAYOUT_LINEAR, "mma": _capi.SCALE_LAYOUT_MMA}
_DT = {torch.bfloat16: _capi.BF16, torch.float32: _capi.FP32, torch.float16: _capi.FP16}
_ORIENT = {"row": _capi.OUT_ROW, "col": _capi.OUT_COL, -1: _capi.OUT_ROW, 0: _capi.OUT_COL}


def build(fast_math: bool = False, force: bool = False) -> str:
    from . import _builder as _b

    return _b.build(fast_math=fast_math, force=force)


def _lib():
    return _capi.load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _view3d(x: torch.Tensor):
    """(x3, G, M, K, ld) for a [M, K] or [G, M, K] tensor whose rows are
    contiguous and whose matrices are back to back (batch stride M * ld)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (the library has no CPU path)")
    if x.dim() == 2:
        x3 = x.unsqueeze(0)
    elif x.dim() == 3:
        x3 = x
    else:
        raise ValueError("expected a 2-D or 3-D tensor, got %d-D" % x.dim())
    G, M, K = x3.shape
    if K > 1 and x3.stride(2) != 1:
        raise ValueError("the last dimension must be contiguous")
    ld = x3.stride(1) if M > 1 else K
    if G > 1 and x3.stride(0) != M * ld:
        raise ValueError("matrices must be stored back to back (batch stride M * ld)")
    return x3, G, M, K, ld


def _params(G, M, K, ld, in_dtype, out_dtype=None, *, mode="none", outer_block_size=0, outer_2d=False,
            inner_2d=False, scale_format="e4m3", stochastic=False, seed=0, step=0, out_mask=_capi.OUT_ROW,
            use_precomputed_outer=False, scale_layout="linear", col_hadamard=False, hadamard_signs=0,
            precomputed_amax=False, sr_global_rows=0, sr_row_offset=0, sr_matrix_offset=0):
    p = _capi.new_params(_lib())
    p.G, p.M, p.K, p.ld = G, M, K, ld
    p.in_dtype = _DT.get(in_dtype, -1)
    p.out_dtype = _DT.get(out_dtype if out_dtype is not None else in_dtype, -1)
    p.mode = _MODES[mode]
    p.outer_block_size = int(outer_block_size)
    p.outer_2d = int(bool(outer_2d))
    p.inner_2d = int(bool(inner_2d))
    p.scale_format = _FMTS[scale_format]
    p.rounding = _capi.STOCHASTIC if stochastic else _capi.RNE
    p.seed = int(seed) & (2 ** 64 - 1)
    p.step = int(step) & (2 ** 32 - 1)
    p.out_mask = int(out_mask)
    p.use_precomputed_outer = int(bool(use_precomputed_outer))
    p.scale_layout = _LAYOUTS[scale_layout]
    p.col_hadamard = int(bool(col_hadamard))
    p.hadamard_signs = int(hadamard_signs) & 0xFFFF
    p.precomputed_amax = int(bool(precomputed_amax))
    p.sr_global_rows, p.sr_row_offset, p.sr_matrix_offset = int(sr_global_rows), int(sr_row_offset), int(sr_matrix_offset)
    return p


def query_sizes(p) -> _capi.Sizes:
    s = _capi.Sizes()
    _capi.check(_lib().fp4q_query_sizes(ctypes.byref(p), ctypes.byref(s)), "fp4q_query_sizes")
    return s


@dataclass
class QuantizedFP4:
    """Outputs of ``quantize``; absent orientations / scales are None."""
    shape: tuple
    mode: str
    outer_block_size: int
    outer_2d: bool
    inner_2d: bool
    scale_format: str
    row_codes: Optional[torch.Tensor] = None   # uint8 [G, M, K/2]
    row_scales: Optional[torch.Tensor] = None  # uint8 [G, M, K/16] (linear layout; flat padded tiles for "mma")
    row_outer: Optional[torch.Tensor] = None   # float32 [G, M, K/ob]
    col_codes: Optional[torch.Tensor] = None   # uint8 [G, K, M/2]
    col_scales: Optional[torch.Tensor] = None  # uint8 [G, K, M/16]
    col_outer: Optional[torch.Tensor] = None   # float32 [G, K, M/ob]
    tile_outer: Optional[torch.Tensor] = None  # float32 [G, M/ob, K/ob] or [1]
    scale_layout: str = "linear"               # inner-scale layout: "linear" or "mma" (128 x 4 tiles)
    group_offsets: Optional[torch.Tensor] = None  # quantize_grouped: int64 [groups + 1]
    group_error: Optional[torch.Tensor] = None    # quantize_grouped: nonzero if the offsets were invalid


def _outer_shapes(G, M, K, mode, ob, outer_2d, row, col):
    shp = {"row_outer": None, "col_outer": None, "tile_outer": None}
    if mode == "tensorwise":
        shp["tile_outer"] = (1,)
    elif mode == "outer_block":
        if outer_2d:
            shp["tile_outer"] = (G, M // ob, K // ob)
        else:
            if row:
                shp["row_outer"] = (G, M, K // ob)
            if col:
                shp["col_outer"] = (G, K, M // ob)
    return shp


def quantize(x: torch.Tensor, *, mode: str = "none", outer_block_size: int = 0, outer_2d: bool = False,
             inner_2d: bool = False, scale_format: str = "e4m3", stochastic: bool = False, seed: int = 0,
             step: int = 0, rowwise: bool = True, columnwise: bool = False,
             residual: Optional[torch.Tensor] = None, precomputed_outer: Optional[QuantizedFP4] = None,
             out: Optional[QuantizedFP4] = None, scale_layout: str = "linear", col_hadamard: bool = False,
             hadamard_signs: int = 0, tensorwise_amax: Optional[torch.Tensor] = None, sr_global_rows: int = 0,
             sr_row_offset: int = 0, sr_matrix_offset: int = 0) -> QuantizedFP4:
    """NVFP4 / AMD-FP4 quantize of a CUDA bf16 or fp32 tensor ([M, K] or [G, M, K]).

    ``residual`` (fp32, [G, M, K] contiguous) enables error feedback and is
    updated in place (rowwise only).  ``precomputed_outer`` supplies outer
    scales (from an earlier call) instead of computing them.  ``out`` reuses
    preallocated output buffers.  ``scale_layout="mma"`` writes the inner
    scales in the 128 x 4 tiled layout block-scaled tensor-core MMAs read
    (see include/fp4q.h); the scale tensors are then flat padded byte
    buffers.  ``col_hadamard`` applies the random Hadamard transform along M
    (16-row blocks, sign mask ``hadamard_signs``) before the columnwise
    quantization.

    ``tensorwise_amax``: a workspace from ``tensorwise_workspace()`` whose
    ``workspace_amax`` already holds the amax of the whole tensor (e.g. the
    maximum over the shards of a tensor split across processes); the
    tensorwise scale is then computed from it on the device.
    ``sr_global_rows`` / ``sr_row_offset`` / ``sr_matrix_offset``: this
    tensor is rows ``sr_row_offset ..`` (of ``sr_global_rows``) and matrices
    ``sr_matrix_offset ..`` of a larger one, whose element positions key the
    stochastic-rounding draws (see include/fp4q.h)."""
    x3, G, M, K, ld = _view3d(x)
    mask = (_capi.OUT_ROW if rowwise else 0) | (_capi.OUT_COL if columnwise else 0)
    p = _params(G, M, K, ld, x.dtype, mode=mode, outer_block_size=outer_block_size, outer_2d=outer_2d,
                inner_2d=inner_2d, scale_format=scale_format, stochastic=stochastic, seed=seed, step=step,
                out_mask=mask, use_precomputed_outer=precomputed_outer is not None, scale_layout=scale_layout,
                col_hadamard=col_hadamard, hadamard_signs=hadamard_signs,
                precomputed_amax=tensorwise_amax is not None, sr_global_rows=sr_global_rows,
                sr_row_offset=sr_row_offset, sr_matrix_offset=sr_matrix_offset)
    s = query_sizes(p)
    dev = x.device
    if out is None:
        u8 = dict(dtype=torch.uint8, device=dev)
        q = QuantizedFP4((G, M, K), mode, outer_block_size, outer_2d, inner_2d, scale_format,
                         scale_layout=scale_layout)
        mma = scale_layout == "mma"
        if rowwise:
            q.row_codes = torch.empty(G, M, K // 2, **u8)
            q.row_scales = torch.empty(int(s.row_scales), **u8) if mma else torch.empty(G, M, K // 16, **u8)
        if columnwise:
            q.col_codes = torch.empty(G, K, M // 2, **u8)
            q.col_scales = torch.empty(int(s.col_scales), **u8) if mma else torch.empty(G, K, M // 16, **u8)
        for name, shp in _outer_shapes(G, M, K, mode, outer_block_size, outer_2d, rowwise, columnwise).items():
            if shp is not None:
                src = getattr(precomputed_outer, name, None) if precomputed_outer is not None else None
                setattr(q, name, src if src is not None else torch.empty(shp, dtype=torch.float32, device=dev))
    else:
        q = out
    o = _capi.Outputs(*[_ptr(getattr(q, n)) for n in
                        ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer",
                         "tile_outer")])
    if tensorwise_amax is not None:
        if tensorwise_amax.dtype != torch.uint8 or tensorwise_amax.numel() < s.workspace or not tensorwise_amax.is_cuda:
            raise ValueError("tensorwise_amax must be a CUDA workspace from tensorwise_workspace()")
        ws = tensorwise_amax
    else:
        ws = torch.empty(max(int(s.workspace), 1), dtype=torch.uint8, device=dev) if s.workspace else None
    st = _lib().fp4_quantize(ctypes.byref(p), _ptr(x3), ctypes.byref(o), _ptr(residual), _ptr(ws),
                             int(s.workspace), _stream(dev))
    _capi.check(st, "fp4_quantize")
    return q


@dataclass
class FP4Operands:
    """Outputs of ``to_fp4_operands``: the same buffers as the QuantizedFP4,
    viewed as torch's FP4 / FP8 dtypes."""
    codes: torch.Tensor       # float4_e2m1fn_x2 [M, K/2] (or [G, M, K/2])
    scales: torch.Tensor      # float8_e4m3fn, flat, 128 x 4 tiled tensor-core layout
    quantized: QuantizedFP4   # the underlying uint8 buffers


def to_fp4_operands(x: torch.Tensor, stochastic: bool = False, seed: int = 0, step: int = 0,
                    residual: Optional[torch.Tensor] = None) -> FP4Operands:
    """NVFP4 quantize of x ([M, K] or [G, M, K], bf16 / fp32) into the operand
    form of torch's block-scaled FP4 matmul (fp4-train README, "API":
    to_fp4_operands, packed fp4 + e4m3 scale as the torch FP4 dtypes for
    ``_scaled_mm``): per-16 E4M3 scales along K in the tensor-core layout,
    codes two per byte.  ``stochastic`` / ``seed`` / ``step`` / ``residual``
    as for ``quantize``.  The views share the quantizer's buffers."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        raise RuntimeError("this torch has no float4_e2m1fn_x2 dtype")
    q = quantize(x, stochastic=stochastic, seed=seed, step=step, residual=residual, scale_layout="mma")
    codes = q.row_codes if x.dim() == 3 else q.row_codes[0]
    return FP4Operands(codes.view(torch.float4_e2m1fn_x2), q.row_scales.view(torch.float8_e4m3fn), q)


def quantize_grouped(x: torch.Tensor, offsets: torch.Tensor, *, mode: str = "none", outer_block_size: int = 0,
                     outer_2d: bool = False, scale_format: str = "e4m3", stochastic: bool = False, seed: int = 0,
                     step: int = 0, rowwise: bool = True, columnwise: bool = False,
                     precomputed_outer: Optional[QuantizedFP4] = None, out: Optional[QuantizedFP4] = None,
                     workspace: Optional[torch.Tensor] = None) -> QuantizedFP4:
    """Ragged grouped NVFP4 / AMD-FP4 quantize: rows offsets[e] ..
    offsets[e + 1] of the bf16 [M, K] CUDA tensor x form group e (e.g. the
    tokens routed to expert e), each quantized as a matrix of its own.
    ``offsets`` is a CUDA int64 tensor [groups + 1] (read on the device).
    Columnwise buffers hold each group's transpose back to back (see
    include/fp4q.h); tensorwise mode gives one scale per group in
    ``tile_outer``.  Invalid offsets write nothing and set ``q.group_error``
    (a CUDA int32 tensor) nonzero."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    if not (offsets.is_cuda and offsets.dtype == torch.int64 and offsets.dim() == 1 and offsets.is_contiguous()):
        raise ValueError("offsets must be a contiguous CUDA int64 vector [groups + 1]")
    x3, G, M, K, ld = _view3d(x)
    ngroups = offsets.numel() - 1
    mask = (_capi.OUT_ROW if rowwise else 0) | (_capi.OUT_COL if columnwise else 0)
    p = _params(G, M, K, ld, x.dtype, mode=mode, outer_block_size=outer_block_size, outer_2d=outer_2d,
                scale_format=scale_format, stochastic=stochastic, seed=seed, step=step, out_mask=mask,
                use_precomputed_outer=precomputed_outer is not None)
    s = _capi.Sizes()
    _capi.check(_lib().fp4q_query_sizes_grouped(ctypes.byref(p), ngroups, ctypes.byref(s)), "fp4q_query_sizes_grouped")
    dev = x.device
    if out is None:
        u8 = dict(dtype=torch.uint8, device=dev)
        q = QuantizedFP4((1, M, K), mode, outer_block_size, outer_2d, False, scale_format)
        if rowwise:
            q.row_codes = torch.empty(1, M, K // 2, **u8)
            q.row_scales = torch.empty(1, M, K // 16, **u8)
        if columnwise:
            q.col_codes = torch.empty(K * M // 2, **u8)      # group transposes back to back
            q.col_scales = torch.empty(K * M // 16, **u8)
        for name, nbytes in (("row_outer", s.row_outer), ("col_outer", s.col_outer), ("tile_outer", s.tile_outer)):
            if nbytes:
                src = getattr(precomputed_outer, name, None) if precomputed_outer is not None else None
                setattr(q, name, src if src is not None else torch.empty(int(nbytes) // 4, dtype=torch.float32,
                                                                          device=dev))
    else:
        q = out
    q.group_offsets = offsets
    if workspace is None or workspace.numel() < s.workspace:
        workspace = torch.empty(int(s.workspace), dtype=torch.uint8, device=dev)
    q.group_error = workspace[:4].view(torch.int32)
    o = _capi.Outputs(*[_ptr(getattr(q, n)) for n in
                        ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer",
                         "tile_outer")])
    st = _lib().fp4_quantize_grouped(ctypes.byref(p), _ptr(x3), _ptr(offsets), ngroups, ctypes.byref(o),
                                     _ptr(workspace), int(workspace.numel()), _stream(dev))
    _capi.check(st, "fp4_quantize_grouped")
    return q


def dequantize(q: QuantizedFP4, orient: str = "row", out_dtype: torch.dtype = torch.bfloat16,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dequantize one orientation of ``q``: [G, M, K] (row) or [G, K, M] (col)."""
    G, M, K = q.shape
    o = _ORIENT[orient]
    codes = q.row_codes if o == _capi.OUT_ROW else q.col_codes
    scales = q.row_scales if o == _capi.OUT_ROW else q.col_scales
    if q.mode == "outer_block" and not q.outer_2d:
        outer = q.row_outer if o == _capi.OUT_ROW else q.col_outer
    else:
        outer = q.tile_outer
    p = _params(G, M, K, K, torch.bfloat16, out_dtype, mode=q.mode, outer_block_size=q.outer_block_size,
                outer_2d=q.outer_2d, inner_2d=q.inner_2d, scale_format=q.scale_format, out_mask=o,
                scale_layout=q.scale_layout)
    R, C = (M, K) if o == _capi.OUT_ROW else (K, M)
    y = out if out is not None else torch.empty(G, R, C, dtype=out_dtype, device=codes.device)
    st = _lib().fp4_dequantize(ctypes.byref(p), o, _ptr(codes), _ptr(scales), _ptr(outer), _ptr(y),
                               _stream(codes.device))
    _capi.check(st, "fp4_dequantize")
    return y


def qdq(x: torch.Tensor, *, axis: int = -1, mode: str = "none", outer_block_size: int = 0,
        outer_2d: bool = False, inner_2d: bool = False, scale_format: str = "e4m3", stochastic: bool = False,
        seed: int = 0, step: int = 0, residual: Optional[torch.Tensor] = None,
        precomputed_outer: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
        out: Optional[torch.Tensor] = None, tensorwise_amax: Optional[torch.Tensor] = None, sr_global_rows: int = 0,
        sr_row_offset: int = 0, sr_matrix_offset: int = 0):
    """Quantize-dequantize along ``axis`` (-1: blocks along K; 0: along M).

    Returns (y, outer) with y [G, M, K] (or [M, K]) in ``out_dtype`` (x's dtype
    by default) and ``outer`` the outer scales used (None in mode none)."""
    x3, G, M, K, ld = _view3d(x)
    o = _ORIENT[axis]
    out_dtype = out_dtype or x.dtype
    p = _params(G, M, K, ld, x.dtype, out_dtype, mode=mode, outer_block_size=outer_block_size,
                outer_2d=outer_2d, inner_2d=inner_2d, scale_format=scale_format, stochastic=stochastic,
                seed=seed, step=step, out_mask=o, use_precomputed_outer=precomputed_outer is not None,
                precomputed_amax=tensorwise_amax is not None, sr_global_rows=sr_global_rows,
                sr_row_offset=sr_row_offset, sr_matrix_offset=sr_matrix_offset)
    s = query_sizes(p)
    dev = x.device
    shp = _outer_shapes(G, M, K, mode, outer_block_size, outer_2d, o == _capi.OUT_ROW, o == _capi.OUT_COL)
    oshape = next((v for v in shp.values() if v is not None), None)
    if precomputed_outer is not None:
        outer = precomputed_outer
    else:
        outer = torch.empty(oshape, dtype=torch.float32, device=dev) if oshape is not None else None
    y = out if out is not None else torch.empty(G, M, K, dtype=out_dtype, device=dev)
    if tensorwise_amax is not None:
        if tensorwise_amax.dtype != torch.uint8 or tensorwise_amax.numel() < s.workspace or not tensorwise_amax.is_cuda:
            raise ValueError("tensorwise_amax must be a CUDA workspace from tensorwise_workspace()")
        ws = tensorwise_amax
    else:
        ws = torch.empty(int(s.workspace), dtype=torch.uint8, device=dev) if s.workspace else None
    st = _lib().fp4_qdq(ctypes.byref(p), o, _ptr(x3), _ptr(y), _ptr(residual), _ptr(outer), _ptr(ws),
                        int(s.workspace), _stream(dev))
    _capi.check(st, "fp4_qdq")
    return (y if x.dim() == 3 or out is not None else y[0]), outer


def mxfp4_fake_quantize(x: torch.Tensor, out_dtype: Optional[torch.dtype] = None,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MXFP4 projection (E2M1 with 1 x 32 power-of-two scales, RNE) of x."""
    x3, G, M, K, ld = _view3d(x)
    out_dtype = out_dtype or x.dtype
    p = _params(G, M, K, ld, x.dtype, out_dtype)
    y = out if out is not None else torch.empty(G, M, K, dtype=out_dtype, device=x.device)
    st = _lib().mxfp4_fake_quantize(ctypes.byref(p), _ptr(x3), _ptr(y), _stream(x.device))
    _capi.check(st, "mxfp4_fake_quantize")
    return y if (x.dim() == 3 or out is not None) else y[0]


@dataclass
class MXFP8Pair:
    """Outputs of mxfp4_project_mxfp8; absent parts are None."""
    y: Optional[torch.Tensor] = None           # the MXFP4 projection [G, M, K]
    row_codes: Optional[torch.Tensor] = None   # E4M3 bytes [G, M, K]
    row_scales: Optional[torch.Tensor] = None  # UE8M0 bytes [G, M, K/32]
    col_codes: Optional[torch.Tensor] = None   # E4M3 bytes [G, K, M]
    col_scales: Optional[torch.Tensor] = None  # UE8M0 bytes [G, K, M/32]


def mxfp4_project_mxfp8(x: torch.Tensor, *, rowwise: bool = True, columnwise: bool = True, with_y: bool = False,
                        out_dtype: Optional[torch.dtype] = None, out: Optional[MXFP8Pair] = None) -> MXFP8Pair:
    """Fused MXFP4 projection of x and its MXFP8 encodings (rowwise 1 x 32,
    columnwise 32 x 1), reading x once; ``with_y`` also returns the
    projection itself.  See include/fp4q.h for the MXFP8 rule."""
    x3, G, M, K, ld = _view3d(x)
    out_dtype = out_dtype or x.dtype
    mask = (_capi.OUT_ROW if rowwise else 0) | (_capi.OUT_COL if columnwise else 0)
    p = _params(G, M, K, ld, x.dtype, out_dtype, out_mask=mask)
    dev = x.device
    if out is None:
        u8 = dict(dtype=torch.uint8, device=dev)
        out = MXFP8Pair()
        if with_y:
            out.y = torch.empty(G, M, K, dtype=out_dtype, device=dev)
        if rowwise:
            out.row_codes, out.row_scales = torch.empty(G, M, K, **u8), torch.empty(G, M, K // 32, **u8)
        if columnwise:
            out.col_codes, out.col_scales = torch.empty(G, K, M, **u8), torch.empty(G, K, M // 32, **u8)
    st = _lib().mxfp4_project_mxfp8(ctypes.byref(p), _ptr(x3), _ptr(out.y), _ptr(out.row_codes), _ptr(out.row_scales),
                                    _ptr(out.col_codes), _ptr(out.col_scales), _stream(dev))
    _capi.check(st, "mxfp4_project_mxfp8")
    return out


HOST_CHUNK_BYTES = 16 << 20


def host_workspace_bytes(K: int, in_dtype: torch.dtype = torch.bfloat16, out_dtype: Optional[torch.dtype] = None) -> int:
    """Device staging bytes mxfp4_fake_quantize_host needs for full-size
    chunks of rows of K elements."""
    out_dtype = out_dtype or in_dtype
    ein, eout = torch.empty(0, dtype=in_dtype).element_size(), torch.empty(0, dtype=out_dtype).element_size()
    rows = max(1, HOST_CHUNK_BYTES // (K * ein))
    r256 = lambda v: (v + 255) // 256 * 256
    return 2 * (r256(rows * K * ein) + r256(rows * K * eout))


def mxfp4_fake_quantize_host(x: torch.Tensor, out_dtype: Optional[torch.dtype] = None,
                             out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                             device=None, synchronize: bool = True) -> torch.Tensor:
    """MXFP4 projection of a tensor in HOST memory (pinned for overlap),
    streamed through the GPU in chunks: host-to-device copy, kernel and
    device-to-host copy of consecutive chunks overlap.  Returns a host
    tensor; with synchronize=False it is complete when the current stream of
    `device` reaches this point."""
    if x.is_cuda:
        raise ValueError("x must be a host tensor (use mxfp4_fake_quantize for device tensors)")
    if x.dim() == 2:
        x3 = x.unsqueeze(0)
    elif x.dim() == 3:
        x3 = x
    else:
        raise ValueError("expected a 2-D or 3-D tensor")
    G, M, K = x3.shape
    if K > 1 and x3.stride(2) != 1:
        raise ValueError("the last dimension must be contiguous")
    ld = x3.stride(1) if M > 1 else K
    if G > 1 and x3.stride(0) != M * ld:
        raise ValueError("matrices must be stored back to back (batch stride M * ld)")
    out_dtype = out_dtype or x.dtype
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    y = out if out is not None else torch.empty(G, M, K, dtype=out_dtype, pin_memory=x.is_pinned())
    if workspace is None:
        workspace = torch.empty(host_workspace_bytes(K, x.dtype, out_dtype), dtype=torch.uint8, device=dev)
    p = _params(G, M, K, ld, x.dtype, out_dtype)
    with torch.cuda.device(dev):
        st = _lib().mxfp4_fake_quantize_host(ctypes.byref(p), ctypes.c_void_p(x3.data_ptr()),
                                             ctypes.c_void_p(y.data_ptr()), _ptr(workspace),
                                             workspace.numel(), _stream(dev))
        _capi.check(st, "mxfp4_fake_quantize_host")
        if synchronize:
            torch.cuda.current_stream(dev).synchronize()
    return y if (x.dim() == 3 or out is not None) else y[0]


TENSORWISE_WORKSPACE_BYTES = 256


def tensorwise_workspace(device) -> torch.Tensor:
    """A device workspace for tensorwise quantization whose first float
    (``workspace_amax``) carries the tensor's amax: fill it with
    ``tensor_amax(x, out=workspace_amax(ws))`` (and, across processes, an
    all-reduce MAX of that float), then pass it as ``tensorwise_amax``."""
    return torch.zeros(TENSORWISE_WORKSPACE_BYTES, dtype=torch.uint8, device=device)


def workspace_amax(ws: torch.Tensor) -> torch.Tensor:
    """The 1-element float32 view of a tensorwise workspace's amax."""
    return ws[:4].view(torch.float32)


def device_status(clear: bool = True, device=None) -> None:
    """Wait for the current stream, then raise FP4QError(FP4Q_ERR_TIMEOUT) if
    a kernel's bounded wait for its tile copy ran out on this device since the
    flags were last cleared (the outputs of that call are not valid)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _capi.check(_lib().fp4q_device_status(int(bool(clear)), _stream(dev)), "fp4q_device_status")


def tensor_amax(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """max |sanitize(x + residual)| over a CUDA bf16 / fp32 tensor, as a
    1-element float32 device tensor (the tensorwise outer scale is this
    value / (scale_max * 6))."""
    x3, G, M, K, ld = _view3d(x)
    p = _params(G, M, K, ld, x.dtype)
    a = out if out is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    st = _lib().fp4_tensor_amax(ctypes.byref(p), _ptr(x3), _ptr(residual), _ptr(a), _stream(x.device))
    _capi.check(st, "fp4_tensor_amax")
    return a
