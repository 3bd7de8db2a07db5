"""Row-sharded quantization across processes, one GPU per process.

Every unit of the method is independent of the others -- 1 x 16 and 16 x 16
inner blocks, 1 x ob and ob x ob outer blocks, 1 x 32 MXFP4 blocks -- so a
tensor split by rows at block boundaries quantizes shard by shard with no
communication ("NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
training", "Technical design": the outer block is the unit of the outer
scale).  The one exception is the tensorwise scale, whose amax spans the
whole tensor ("Background": the per-tensor scale): each process computes
its shard's amax, one all-reduce (MAX) of a single float combines them, and
every shard is quantized with S = amax / (scale_max * 6) passed as a
precomputed tensorwise scale.  The maximum is exact and S is the same
binary32 division the single-process path does, so the shards' codes and
scales are bit-identical to slices of the unsharded result.

Stochastic rounding draws from the element's index within the tensor that
is being quantized; a shard is quantized as a tensor of its own, so its
random stream is keyed by shard-local indices (deterministic, with the same
statistics, but not the unsharded stream).
"""
from __future__ import annotations

import math
from typing import Optional

import torch
import torch.distributed as dist

from . import QuantizedFP4, quantize, tensor_amax

# scale_max * 6 of each inner-scale format (E4M3: 448 * 6, UE5M3: 114688 * 6)
DENOM = {"e4m3": 2688.0, "ue5m3": 688128.0}


def shard_alignment(mode: str = "none", outer_block_size: int = 0, outer_2d: bool = False,
                    columnwise: bool = False, inner_2d: bool = False) -> int:
    """Row multiple at which a tensor may be split so that no block of the
    requested outputs straddles two shards."""
    a = 1
    if columnwise or inner_2d:
        a = 16  # columnwise / 16 x 16 inner blocks span 16 rows
    if mode == "outer_block" and (outer_2d or columnwise):
        a = a * outer_block_size // math.gcd(a, outer_block_size)
    return a


def row_range(M: int, world: int, rank: int, align: int = 1):
    """Rows [lo, hi) of `rank` when M rows are cut into `world` contiguous
    shards whose boundaries are multiples of `align` (sizes differ by at most
    one unit of `align`; trailing ranks may get no rows)."""
    if world < 1 or not 0 <= rank < world or align < 1:
        raise ValueError("bad world / rank / align")
    units = -(-M // align)
    per, extra = divmod(units, world)
    lo = rank * per + min(rank, extra)
    hi = lo + per + (1 if rank < extra else 0)
    return min(lo * align, M), min(hi * align, M)


def tensorwise_scale(local_amax: torch.Tensor, scale_format: str = "e4m3", group=None) -> torch.Tensor:
    """The tensorwise outer scale of a row-sharded tensor from this process's
    shard amax (1-element float32): all-reduce MAX over `group`, then one
    binary32 division by scale_max * 6."""
    a = local_amax.detach().to(torch.float32).reshape(1).clone()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(a, op=dist.ReduceOp.MAX, group=group)
    return a / DENOM[scale_format]


def quantize_shard(x_local: torch.Tensor, *, group=None, mode: str = "none", scale_format: str = "e4m3",
                   residual: Optional[torch.Tensor] = None, **kw) -> QuantizedFP4:
    """Quantize this process's row shard of a tensor split across the
    processes of `group` (boundaries at multiples of shard_alignment(...)).
    Outer-block and none modes run locally; tensorwise mode first agrees on
    the global scale (tensorwise_scale)."""
    if mode != "tensorwise":
        return quantize(x_local, mode=mode, scale_format=scale_format, residual=residual, **kw)
    S = tensorwise_scale(tensor_amax(x_local, residual), scale_format, group)
    shape = tuple(x_local.shape) if x_local.dim() == 3 else (1,) + tuple(x_local.shape)
    pre = QuantizedFP4(shape, "tensorwise", 0, False, bool(kw.get("inner_2d", False)), scale_format, tile_outer=S)
    return quantize(x_local, mode="tensorwise", scale_format=scale_format, residual=residual,
                    precomputed_outer=pre, **kw)
