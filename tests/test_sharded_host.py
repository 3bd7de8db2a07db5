"""Host logic of the multi-process path, on CPU: the row split, the
tensorwise-scale all-reduce between two gloo ranks, and bench.py's rank
barrier / max-over-ranks timing.  No GPU: the shard amax is computed here
with numpy from the sanitizing rule (NaN -> +0, +-inf -> +-largest finite)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from block_scaled_fp4_quantize_gb300 import sharded
from block_scaled_fp4_quantize_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _np_amax_bf16(x: torch.Tensor) -> float:
    a = np.abs(x.float().numpy().astype(np.float64))
    a[np.isnan(a)] = 0.0
    a[np.isinf(a)] = float(torch.finfo(torch.bfloat16).max)
    return float(a.max()) if a.size else 0.0


def test_row_range_covers_rows_once():
    for M, world, align in ((16384, 2, 1), (16384, 3, 64), (100, 4, 16), (5760, 8, 128), (0, 2, 16), (48, 4, 16)):
        seen = []
        for r in range(world):
            lo, hi = sharded.row_range(M, world, r, align)
            assert 0 <= lo <= hi <= M
            assert lo % align == 0 and (hi % align == 0 or hi == M)
            seen.extend(range(lo, hi))
        assert seen == list(range(M))
    with pytest.raises(ValueError):
        sharded.row_range(16, 0, 0)


def test_shard_alignment():
    assert sharded.shard_alignment() == 1
    assert sharded.shard_alignment("outer_block", 64) == 1          # 1 x 64 rowwise blocks lie in a row
    assert sharded.shard_alignment("outer_block", 64, columnwise=True) == 64
    assert sharded.shard_alignment("outer_block", 48, outer_2d=True) == 48
    assert sharded.shard_alignment("outer_block", 48, columnwise=True) == 48
    assert sharded.shard_alignment("none", columnwise=True) == 16
    assert sharded.shard_alignment("tensorwise", inner_2d=True) == 16


def _tensorwise_worker(rank, world, port, amax_expected):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        x = W.activations(M=512, K=256, n_cols=3, n_rows=1)
        x.view(-1)[7] = float("nan")
        x.view(-1)[300 * 256 + 5] = float("inf")  # in rank 1's rows
        lo, hi = sharded.row_range(x.shape[0], world, rank, 16)
        local = torch.tensor([_np_amax_bf16(x[lo:hi])], dtype=torch.float32)
        a = sharded.allreduce_amax(local)
        assert a is local and a.dtype == torch.float32 and a.shape == (1,)
        assert a.view(torch.int32).item() == np.float32(amax_expected).view(np.int32), (rank, a.item(), amax_expected)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt,denom", [("e4m3", 2688.0), ("ue5m3", 688128.0)])
def test_tensorwise_amax_allreduce_two_ranks(orc, fmt, denom):
    """The all-reduced shard amax is the whole tensor's, bit for bit, on both
    ranks: divided by scale_max * 6 it gives the oracle's tensorwise scale
    of the whole tensor (the library does that division on the device)."""
    x = W.activations(M=512, K=256, n_cols=3, n_rows=1)
    x.view(-1)[7] = float("nan")
    x.view(-1)[300 * 256 + 5] = float("inf")
    xb = x.view(torch.int16).numpy().view(np.uint16)[None]
    ref = orc.quantize(xb, mode="tensorwise", fmt=fmt, out_mask=1)
    amax = np.float32(_np_amax_bf16(x))
    assert (amax / np.float32(denom)).view(np.uint32) == ref["tile_outer"].reshape(-1)[0].view(np.uint32)
    mp.spawn(_tensorwise_worker, args=(2, _free_port(), float(amax)), nprocs=2, join=True)


def _bench_dist_worker(rank, world, port):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    d = bench.Dist()
    try:
        assert d.world == world and d.rank == rank
        d.barrier()
        assert d.max(1.5 + rank) == 1.5 + world - 1
        assert d.max(-float(rank)) == 0.0
    finally:
        d.close()


def test_bench_dist_two_ranks():
    """bench.py's timing takes the maximum over ranks after a barrier."""
    mp.spawn(_bench_dist_worker, args=(2, _free_port()), nprocs=2, join=True)
