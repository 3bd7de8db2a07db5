"""Seeded synthetic inputs shaped like the quantizer's workloads.

This module only draws random numbers and places edge values; it holds none
of the quantizer's arithmetic, so both the CUDA path's tests/benchmark and the
CPU oracle can take their inputs from it.  Every generator is deterministic in
its seeds and returns CPU tensors (bf16 data as ``torch.bfloat16``).

Workloads (shapes and value distributions of the pages' use cases):

* ``small_nvfp4``   bf16 [256, 512] ~ N(0, 1), seed 0 (NVFP4 quantize with 1x64
  outer blocks, then dequantize).
* ``mxfp4_weight``  bf16 [8192, 8192] ~ N(0, 0.02), seed 0, with 0.1 % of the
  1x32 blocks overwritten by edge patterns (randperm seed 1), plus a
  [256, 256] tensor holding every bf16 bit pattern.
* ``activations``   bf16 [16384, 2880] ~ N(0, 1), seed 0; 14 columns (0.5 %,
  randperm seed 1) x 1e3 and 2 rows (0.01 %, randperm seed 2) x 1e2 --
  "massive activations" at the GPT-OSS hidden width.
* ``moe_experts``   bf16 [32, 5760, 2880]: expert e ~ N(0, 0.02) from seed e,
  with entries where U(0,1) < 0.01 (seed 1000 + e) multiplied by 200.
* ``sr_ef_weight``  fp32 [8192, 8192] ~ N(0, 0.02), seed 0, residual 0; the
  per-step gradient of step t is N(0, 1) from seed 1000 + t.
"""
from __future__ import annotations

import numpy as np
import torch

MXFP4_EDGE_PATTERNS = (
    "signed_zero", "sub_2m127", "sub_2m128", "sub_2m133", "pos_inf", "nan",
    "cap", "cap_plus_ulp", "rne_midpoints", "threshold_below", "threshold_at", "threshold_above",
)


def _randn(shape, seed, std=1.0, dtype=torch.float32):
    g = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def small_nvfp4():
    """bf16 [256, 512] ~ N(0, 1), seed 0."""
    return _randn((256, 512), 0).to(torch.bfloat16)


def bf16_bits(v):
    """Bit pattern of float ``v`` (exactly representable in bf16)."""
    b = np.array([v], np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, "value is not a bf16"
    return int(b >> 16)


def _edge_block(kind, rng):
    """One 32-element block (uint16 bf16 bits) of the named edge pattern."""
    sign = rng.integers(0, 2, 32).astype(np.uint16) << 15
    if kind == "signed_zero":
        return sign.copy()
    if kind in ("sub_2m127", "sub_2m128", "sub_2m133"):
        e = {"sub_2m127": 127, "sub_2m128": 128, "sub_2m133": 133}[kind]
        mag = np.uint16(1 << (133 - e))  # bf16 subnormal 2^-e = (1 << (133-e)) * 2^-133
        return (sign | mag).astype(np.uint16)
    k = int(rng.integers(-20, 21))
    base = (rng.standard_normal(32) * 2.0 ** k).astype(np.float32)
    bits = (base.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    pos = int(rng.integers(0, 32))
    if kind == "pos_inf":
        bits[pos] = 0x7F80
    elif kind == "nan":
        bits[pos] = 0x7FC1
    elif kind == "cap":
        bits = (bits & 0x8000) | np.minimum(bits & 0x7FFF, 0x7F00).astype(np.uint16)
        bits[pos] = bf16_bits(6.0 * 2.0 ** 125)
    elif kind == "cap_plus_ulp":
        bits = (bits & 0x8000) | np.minimum(bits & 0x7FFF, 0x7F00).astype(np.uint16)
        bits[pos] = bf16_bits(6.0 * 2.0 ** 125) + 1
    elif kind == "rne_midpoints":
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
        vals = mids[rng.integers(0, 7, 32)] * np.float32(2.0 ** k)
        vals[pos] = np.float32(6.0 * 2.0 ** k)
        bits = (vals.view(np.uint32) >> 16).astype(np.uint16) | sign
    elif kind.startswith("threshold"):
        # block maximum one bf16 ulp below, at, or one ulp above 6 * 2^k
        at = bf16_bits(6.0 * 2.0 ** k)
        top = {"threshold_below": at - 1, "threshold_at": at, "threshold_above": at + 1}[kind]
        small = (np.abs(base) * np.float32(0.25)).astype(np.float32)
        bits = (small.view(np.uint32) >> 16).astype(np.uint16) | sign
        bits[pos] = np.uint16(top) | sign[pos]
    return bits.astype(np.uint16)


def mxfp4_weight(M=8192, K=8192, frac=0.001, seed=0, edge_seed=1):
    """bf16 [M, K] ~ N(0, 0.02) with edge blocks; returns (x, edge_block_ids)."""
    x = _randn((M, K), seed, 0.02).to(torch.bfloat16)
    nblk = M * K // 32
    n_edge = int(nblk * frac)
    g = torch.Generator("cpu").manual_seed(edge_seed)
    ids = torch.randperm(nblk, generator=g)[:n_edge].numpy()
    rng = np.random.default_rng(edge_seed)
    bits = x.view(torch.int16).numpy().view(np.uint16).reshape(-1, 32)
    for n, b in enumerate(ids):
        bits[b] = _edge_block(MXFP4_EDGE_PATTERNS[n % len(MXFP4_EDGE_PATTERNS)], rng)
    return x, ids


def all_bf16_patterns():
    """bf16 [256, 256]; element (r, c) has bit pattern 256 r + c."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)


def activations(M=16384, K=2880, seed=0, n_cols=None, n_rows=None):
    """bf16 [M, K] ~ N(0, 1) with massive-activation columns (x1e3) and rows (x1e2)."""
    x = _randn((M, K), seed)
    n_cols = max(1, round(0.005 * K)) if n_cols is None else n_cols
    n_rows = max(1, round(0.0001 * M)) if n_rows is None else n_rows
    cols = torch.randperm(K, generator=torch.Generator("cpu").manual_seed(1))[:n_cols]
    rows = torch.randperm(M, generator=torch.Generator("cpu").manual_seed(2))[:n_rows]
    x[:, cols] *= 1e3
    x[rows, :] *= 1e2
    return x.to(torch.bfloat16)


def moe_expert(e, M=5760, K=2880):
    """bf16 [M, K]: expert e ~ N(0, 0.02) (seed e), 1 % outliers x 200 (seed 1000 + e)."""
    x = _randn((M, K), e, 0.02)
    g = torch.Generator("cpu").manual_seed(1000 + e)
    mask = torch.rand(M, K, generator=g) < 0.01
    x[mask] *= 200.0
    return x.to(torch.bfloat16)


def moe_experts(G=32, M=5760, K=2880, experts=None):
    experts = range(G) if experts is None else experts
    return torch.stack([moe_expert(e, M, K) for e in experts])


def sr_ef_weight(M=8192, K=8192, seed=0):
    """fp32 [M, K] ~ N(0, 0.02) and a zero fp32 residual of the same shape."""
    return _randn((M, K), seed, 0.02), torch.zeros(M, K, dtype=torch.float32)


def sr_ef_gradient(t, M=8192, K=8192, device="cpu"):
    """Gradient of step t: N(0, 1) from a generator seeded 1000 + t on ``device``."""
    g = torch.Generator(device).manual_seed(1000 + t)
    return torch.randn(M, K, generator=g, device=device, dtype=torch.float32)


def uniform_bf16(shape, seed, lo=-4.0, hi=4.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.rand(*shape, generator=g) * (hi - lo) + lo).to(torch.bfloat16)


def lognormal(shape, seed, sigma=2.0, dtype=torch.bfloat16):
    """Heavy-tailed magnitudes with random signs."""
    g = torch.Generator("cpu").manual_seed(seed)
    mag = torch.exp(torch.randn(*shape, generator=g) * sigma)
    sgn = torch.where(torch.rand(*shape, generator=g) < 0.5, -1.0, 1.0)
    return (mag * sgn).to(dtype)


def large_rows(M, K, seed, device="cuda", chunk_rows=16384):
    """bf16 [M, K] on ``device``: row r ~ N(0, 1) * 2^((r mod 16) - 8), drawn
    in slabs of ``chunk_rows`` rows from one generator seeded ``seed`` (for
    tensors too large to build on the host)."""
    g = torch.Generator(device).manual_seed(seed)
    x = torch.empty(M, K, dtype=torch.bfloat16, device=device)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        sc = torch.exp2(torch.arange(r0, r1, device=device, dtype=torch.float32).remainder(16) - 8.0)
        x[r0:r1] = (torch.randn(r1 - r0, K, generator=g, device=device, dtype=torch.float32) * sc[:, None]).to(torch.bfloat16)
    return x
