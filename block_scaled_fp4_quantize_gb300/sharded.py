"""Row-sharded quantization across processes, one GPU per process.

Every unit of the method is independent of the others -- 1 x 16 and 16 x 16
inner blocks, 1 x ob and ob x ob outer blocks, 1 x 32 MXFP4 blocks -- so a
tensor split by rows at block boundaries quantizes shard by shard with no
communication ("NVFP4 / AMD-FP4 outer-block (two-level) scaling for FP4
training", "Technical design": the outer block is the unit of the outer
scale).  The one exception is the tensorwise scale, whose amax spans the
whole tensor ("Background": the per-tensor scale): each process computes
its shard's amax into a tensorwise workspace, one all-reduce (MAX) of that
single float combines them, and every shard is quantized from the combined
amax, the library dividing it by scale_max * 6 on the device.  The maximum
is exact and the division is the one the single-process path does, so the
shards' codes and scales are bit-identical to slices of the unsharded
result.

Stochastic rounding keys each draw on the element's global index ("fp4-train"
README, "Method": (seed, step, global-index)): a shard passes its first row
and the tensor's row count, so its draws -- and its codes -- are those of the
unsharded tensor in both orientations.
"""
from __future__ import annotations

import math
from typing import Optional

import torch
import torch.distributed as dist

from . import QuantizedFP4, quantize, tensor_amax, tensorwise_workspace, workspace_amax


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


def allreduce_amax(amax: torch.Tensor, group=None) -> torch.Tensor:
    """All-reduce (MAX) a shard's 1-element float32 amax in place over
    `group` (no-op without an initialized multi-process group)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def quantize_shard(x_local: torch.Tensor, *, group=None, mode: str = "none", residual: Optional[torch.Tensor] = None,
                   row_offset: int = 0, global_rows: int = 0, **kw) -> QuantizedFP4:
    """Quantize this process's row shard, rows [row_offset, row_offset +
    x_local.shape[-2]) of a tensor of `global_rows` rows split across the
    processes of `group` (boundaries at multiples of shard_alignment(...)).
    Outer-block and none modes run locally; tensorwise mode first agrees on
    the tensor's amax (one all-reduce of a float).  With stochastic rounding
    the draws follow the rows' global positions (give `global_rows`)."""
    sr = dict(sr_global_rows=global_rows, sr_row_offset=row_offset) if global_rows else {}
    if mode != "tensorwise":
        return quantize(x_local, mode=mode, residual=residual, **sr, **kw)
    ws = tensorwise_workspace(x_local.device)
    a = workspace_amax(ws)
    tensor_amax(x_local, residual, out=a)
    allreduce_amax(a, group)
    return quantize(x_local, mode="tensorwise", residual=residual, tensorwise_amax=ws, **sr, **kw)
