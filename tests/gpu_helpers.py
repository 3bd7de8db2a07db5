"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same host bytes and compare their outputs bit for bit."""
import functools
import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np
import torch

import block_scaled_fp4_quantize_gb300 as fq

ROW, COL = 1, 2


def host_np(t: torch.Tensor) -> np.ndarray:
    """Numpy copy of a CPU/CUDA tensor; bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_kw(kw):
    """Translate binding keyword arguments to the oracle's."""
    o = {}
    o["mode"] = kw.get("mode", "none")
    o["ob"] = kw.get("outer_block_size", 0)
    o["outer_2d"] = kw.get("outer_2d", False)
    o["inner_2d"] = kw.get("inner_2d", False)
    o["fmt"] = kw.get("scale_format", "e4m3")
    o["rounding"] = "sr" if kw.get("stochastic", False) else "rne"
    o["seed"] = kw.get("seed", 0)
    o["step"] = kw.get("step", 0)
    return o


def gpu_quantize(x_cpu, residual_cpu=None, **kw):
    x = x_cpu.cuda()
    r = residual_cpu.cuda() if residual_cpu is not None else None
    q = fq.quantize(x, residual=r, **kw)
    torch.cuda.synchronize()
    out = {}
    for k in ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer"):
        v = getattr(q, k)
        out[k] = None if v is None else host_np(v)
    if r is not None:
        out["residual"] = host_np(r)
    return q, out


def oracle_quantize(orc, x_cpu, residual_cpu=None, **kw):
    x = host_np(x_cpu)
    if x.ndim == 2:
        x = x[None]
    mask = (ROW if kw.get("rowwise", True) else 0) | (COL if kw.get("columnwise", False) else 0)
    r = None if residual_cpu is None else host_np(residual_cpu).copy().reshape(x.shape[0], x.shape[1], -1)
    out = orc.quantize(x, residual=r, out_mask=mask, **oracle_kw(kw))
    if r is not None:
        out["residual"] = r
    return out


def assert_same(gpu: dict, ref: dict, keys=None):
    keys = keys or [k for k in ref if ref[k] is not None]
    for k in keys:
        g, r = gpu.get(k), ref[k]
        assert g is not None, "missing GPU output %s" % k
        g = np.asarray(g).reshape(r.shape)
        if r.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        bad = np.flatnonzero(g.ravel() != r.ravel())
        assert bad.size == 0, "%s: %d of %d differ; first at %d: gpu %r oracle %r" % (
            k, bad.size, r.size, bad[0], g.ravel()[bad[0]], r.ravel()[bad[0]])


def snr_db(x: np.ndarray, y: np.ndarray) -> float:
    x = x.astype(np.float64)
    e = x - y.astype(np.float64)
    return float(10.0 * np.log10((x * x).sum() / (e * e).sum()))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def to_mma_layout(lin: np.ndarray) -> np.ndarray:
    """[G, R, C16] linear inner scales -> the flat 128 x 4 tiled layout that
    block-scaled tensor-core MMAs read (rows padded to 128, columns to 4,
    padding zero; tiles row-major; inside a tile byte (r, c) at
    (r mod 32) * 16 + (r // 32) * 4 + c), written from its definition."""
    G, R, C = lin.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    pad = np.zeros((G, Rp, Cp), np.uint8)
    pad[:, :R, :C] = lin
    t = pad.reshape(G, Rp // 128, 4, 32, Cp // 4, 4)          # g, tile row, r // 32, r % 32, tile col, c
    return np.ascontiguousarray(t.transpose(0, 1, 4, 3, 2, 5)).reshape(-1)


MOE_KW = dict(mode="outer_block", outer_block_size=64, outer_2d=True, rowwise=True, columnwise=True)


def _moe_expert_oracle(args):
    """Worker: the oracle's quantize of MoE expert e (2-D 64 x 64 outer
    scales, both orientations) in scale format fmt."""
    e, fmt = args
    import oracle
    from block_scaled_fp4_quantize_gb300 import workloads as W

    x = host_np(W.moe_expert(e))[None]
    r = oracle.quantize(x, out_mask=ROW | COL, **oracle_kw(dict(MOE_KW, scale_format=fmt)))
    return e, {k: v for k, v in r.items() if v is not None}


@functools.lru_cache(maxsize=2)
def moe_oracle(fmt: str, experts: int = 32):
    """The oracle's outputs for every expert of the MoE workload, computed
    once per format by a pool of spawned processes over the host cores
    (spawned, not forked: the parent process holds a CUDA context)."""
    workers = max(1, min(experts, os.cpu_count() or 1, 16))
    with ProcessPoolExecutor(max_workers=workers, mp_context=multiprocessing.get_context("spawn")) as ex:
        return dict(ex.map(_moe_expert_oracle, [(e, fmt) for e in range(experts)]))
