#!/usr/bin/env python
"""Throughput benchmark of the block-scaled FP4 quantizer on GB300.

One step = one pass of the quantizer over one batch of synthetic input.  The
headline workload is MXFP4 fake-quantization of a bf16 [8192, 8192] weight
~ N(0, 0.02) with 0.1 % edge blocks (the workload the pages quote their
B200 timing on); the metric is GB/s of algorithmic bytes (bf16 in + bf16 out)
and its fraction of the measured HBM copy bandwidth.  The other workloads
(NVFP4 rowwise+columnwise activations, MoE expert weights with 2-D outer
scales, the SR + error-feedback weight update, dequantize) are timed in the
same run and reported under "kernels".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (weak scaling, no data-path collective); timing is bracketed by barriers
and the maximum over ranks is reported by rank 0.  ``--impl reference`` times
the CPU oracle (the plain restatement of the method) on the host cores.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MXFP4_BYTES = 2 * 2 * 8192 * 8192           # bf16 in + bf16 out
B200_CUTE_DSL_GBS = MXFP4_BYTES / 59e-6 / 1e9  # the pages' best figure for this workload (B200)
L2_BYTES = 126 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=25000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-kernel table of other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--only", default=None,
                    help="time only this named non-headline workload (--steps iterations) and print its record")
    ap.add_argument("--experts", type=int, default=32, help="expert count of the MoE workload with --only")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (barriers and a max over ranks only)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        import torch

        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = list(csv.reader(io.StringIO(out)))
        sm, mx, reasons, n_all = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            n_all += 1
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except ValueError:
                continue
            if ts < int(t0) or ts > t1 + 1:
                continue
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except ValueError:
                continue
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# measured peak and ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source has not changed since the counters were taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    ent = table.get(kernel_key)
    if not ent:
        return None
    h = hashlib.sha256()
    for src in ent["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return ent["dram_bytes_per_launch"] if h.hexdigest()[:16] == ent["source_sha256_16"] else None


# ---------------------------------------------------------------------------
# workloads (CUDA path)
# ---------------------------------------------------------------------------

def _warm(fn, warmup, min_seconds=0.5):
    """At least `warmup` calls, and calls for at least `min_seconds`, so the
    GPU's clocks and the memory system reach steady state right before the
    timed region (no idle gap follows)."""
    import torch

    i = 0
    t0 = time.perf_counter()
    while i < warmup or time.perf_counter() - t0 < min_seconds:
        fn(i)
        i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    return i


def graph_split(n, chunk=100):
    """(head, body replays, body size, tail) of n calls: head = min(n,
    chunk) calls, then `body replays` x `body size` calls, then a tail of
    1 .. chunk calls (0 when n <= chunk); the parts add up to n."""
    ch = max(1, min(n, chunk))
    rest = n - ch
    nb = (rest - 1) // ch if rest > 0 else 0
    return ch, nb, ch, rest - nb * ch


class StepGraph:
    """`fn(i)` for i = 0 .. n-1 captured as CUDA graphs (a head graph of up to
    `chunk` calls, a body graph of `chunk` calls replayed as often as needed,
    a tail graph of the rest), so that exactly n calls run.  The replays
    enqueue the same kernels the eager calls do, without the Python launch
    path between them (host-side hiccups then cannot leave the GPU idle
    inside the timed region).  The two timing events are nodes of the head
    and tail graphs (external events): the region they bound is the n
    calls' execution on the GPU, not the host's submission of the first
    graph to an idle GPU.  Where the events cannot be captured they are
    recorded around the replays (`inside` False); where nothing can be
    captured the calls run eagerly (`ok` False)."""

    def __init__(self, fn, n, chunk=100):
        import torch

        self.fn, self.n, self.ok, self.inside = fn, n, False, False
        # head: calls 0 .. h-1; body: `nb` replays of `chunk` calls; tail: the rest (>= 1 when n > chunk)
        self.h, self.nb, self.chunk, self.t = graph_split(n, chunk)
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for i in range(3):
                    fn(i)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            try:
                self.e0 = torch.cuda.Event(enable_timing=True, external=True)
                self.e1 = torch.cuda.Event(enable_timing=True, external=True)
                self._capture(True)
                self.inside = True
            except Exception:  # noqa: BLE001 -- no event nodes in graphs here: events around the replays
                torch.cuda.synchronize()
                self.e0, self.e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                self._capture(False)
            torch.cuda.synchronize()
            self.ok = True
        except Exception as e:  # noqa: BLE001 -- any capture failure falls back to eager calls
            self.error = repr(e)[:200]
            torch.cuda.synchronize()
            self.e0, self.e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def _capture(self, events):
        import torch

        def graph(first, count, head, tail):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if head and events:
                    self.e0.record()
                for i in range(count):
                    self.fn(first + i)
                if tail and events:
                    self.e1.record()
            return g

        self.gh = graph(0, self.h, True, self.t == 0)
        self.gb = graph(self.h, self.chunk, False, False) if self.nb else None
        self.gt = graph(self.h + self.nb * self.chunk, self.t, False, True) if self.t else None

    def run(self):
        if not self.ok:
            for i in range(self.n):
                self.fn(i)
            return
        self.gh.replay()
        for _ in range(self.nb):
            self.gb.replay()
        if self.gt is not None:
            self.gt.replay()

    def timed(self):
        """Run the n calls as the timed region; ms of the region (call after
        a device synchronize)."""
        import torch

        if not (self.ok and self.inside):
            self.e0.record()
        self.run()
        if not (self.ok and self.inside):
            self.e1.record()
        torch.cuda.synchronize()
        return self.e0.elapsed_time(self.e1)


def _events_time(fn, iters, warmup, graph=True):
    """Average ms per call of fn(i) with CUDA events on the current stream,
    over `iters` calls after a warm-up; the calls run as CUDA graph replays
    when they can be captured."""
    import torch

    sg = StepGraph(fn, iters) if graph else None
    if sg is not None and sg.ok:
        _warm(lambda i: sg.run(), 1, min_seconds=0.3)
        torch.cuda.synchronize()
        return sg.timed() / iters
    _warm(fn, warmup, min_seconds=0.3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(iters):
        fn(i)
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def _sets_for(nbytes):
    return max(1, -(-2 * L2_BYTES // max(1, nbytes)))  # enough rotating copies to exceed L2 twice


def _extra_workloads():
    """Named workloads other than the headline, each a function
    (iters, warmup, opts) -> (description, algorithmic bytes, ms per call,
    kernel launches per call).  Kernel only, inputs resident in HBM."""
    import torch

    import block_scaled_fp4_quantize_gb300 as fq
    from block_scaled_fp4_quantize_gb300 import workloads as W

    dev = torch.device("cuda")

    def small_nvfp4_quantize(iters, warmup, opts):
        x = W.small_nvfp4().to(dev)
        q = fq.quantize(x, mode="outer_block", outer_block_size=64)
        ms = _events_time(lambda i: fq.quantize(x, mode="outer_block", outer_block_size=64, out=q), iters, warmup)
        return "bf16[256,512] 1x64 outer E4M3 RNE rowwise", 262144 + 65536 + 8192 + 8192, ms, 1

    def _activations(mode_kw, nb_out, launches, columnwise=True):
        def run(iters, warmup, opts):
            xs = [W.activations().to(dev)]
            nb_in = xs[0].numel() * 2
            for _ in range(_sets_for(nb_in) - 1):
                xs.append(xs[0].clone())
            qs = [fq.quantize(xx, rowwise=True, columnwise=columnwise, **mode_kw) for xx in xs]
            ms = _events_time(lambda i: fq.quantize(xs[i % len(xs)], rowwise=True, columnwise=columnwise,
                                                    out=qs[i % len(xs)], **mode_kw), iters, warmup)
            what = ", ".join("%s=%s" % kv for kv in mode_kw.items() if kv[0] != "mode")
            return ("bf16[16384,2880] massive activations, %s%s, %s" % (
                mode_kw["mode"], " " + what if what else "", "rowwise+columnwise" if columnwise else "rowwise"),
                nb_in + nb_out, ms, launches)
        return run

    M, K = 16384, 2880
    codes = M * K // 2

    def activations_tensorwise(iters, warmup, opts):
        # the whole call (zero the amax word, amax pass, quantize pass) and
        # its two passes timed apart: the amax pass into a workspace, and the
        # quantize pass from that workspace's amax
        run = _activations(dict(mode="tensorwise"), 2 * codes + 2 * (M * K // 16) + 4, 3)
        desc, nb, ms, launches = run(iters, warmup, opts)
        xs = [W.activations().to(dev)]
        for _ in range(_sets_for(xs[0].numel() * 2) - 1):
            xs.append(xs[0].clone())
        wss = [fq.tensorwise_workspace(dev) for _ in xs]
        qs = [fq.quantize(xx, rowwise=True, columnwise=True, mode="tensorwise") for xx in xs]
        n = len(xs)
        ms_amax = _events_time(lambda i: fq.tensor_amax(xs[i % n], out=fq.workspace_amax(wss[i % n])), iters, warmup)
        ms_q = _events_time(lambda i: fq.quantize(xs[i % n], rowwise=True, columnwise=True, mode="tensorwise",
                                                  tensorwise_amax=wss[i % n], out=qs[i % n]), iters, warmup)
        return desc, nb, ms, launches, {"amax_pass_us": round(ms_amax * 1e3, 3),
                                        "quantize_from_amax_us": round(ms_q * 1e3, 3)}

    def dequantize_activations(iters, warmup, opts):
        x = W.activations().to(dev)
        nb = codes + M * K // 16 + M * K // 64 * 4 + M * K * 2
        # rotating sets of (codes, scales, S) and outputs, together above L2
        qds = [fq.quantize(x, mode="outer_block", outer_block_size=64) for _ in range(_sets_for(nb))]
        yds = [torch.empty(1, M, K, dtype=torch.bfloat16, device=dev) for _ in qds]
        ms = _events_time(lambda i: fq.dequantize(qds[i % len(qds)], "row", torch.bfloat16, out=yds[i % len(qds)]),
                          iters, warmup)
        return "codes+scales+S of bf16[16384,2880] -> bf16", nb, ms, 1

    def _moe(fmt):
        def run(iters, warmup, opts):
            G, Me, Ke = opts.get("experts", 32), 5760, 2880
            g = torch.Generator(dev).manual_seed(0)
            xe = torch.randn(G, Me, Ke, generator=g, device=dev) * 0.02
            xe = torch.where(torch.rand(G, Me, Ke, generator=g, device=dev) < 0.01, xe * 200, xe).to(torch.bfloat16)
            kw = dict(mode="outer_block", outer_block_size=64, outer_2d=True, scale_format=fmt, rowwise=True,
                      columnwise=True)
            qe = fq.quantize(xe, **kw)
            ms = _events_time(lambda i: fq.quantize(xe, out=qe, **kw), iters, warmup)
            nb = G * Me * Ke * 2 + 2 * (G * Me * Ke // 2) + 2 * (G * Me * Ke // 16) + G * (Me // 64) * (Ke // 64) * 4
            return "%d x bf16[5760,2880] 2-D 64x64 outer %s rowwise+columnwise" % (G, fmt), nb, ms, 1
        return run

    def mxfp4_project_mxfp8(iters, warmup, opts):
        # the headline weight: projection + MXFP8 rowwise and columnwise in one pass
        xh, _ = W.mxfp4_weight()
        xs = [xh.to(dev) for _ in range(2)]
        outs = [fq.mxfp4_project_mxfp8(xx) for xx in xs]
        ms = _events_time(lambda i: fq.mxfp4_project_mxfp8(xs[i & 1], out=outs[i & 1]), iters, warmup)
        n = xh.numel()
        return ("bf16[8192,8192] -> MXFP4 projection -> MXFP8 rowwise + columnwise (E4M3 + UE8M0)",
                2 * n + 2 * n + 2 * (n // 32), ms, 1)

    def moe_grouped_tokens(iters, warmup, opts):
        # 65536 tokens routed to 32 experts with lognormal popularity (seed 0),
        # each expert's count rounded down to a multiple of 64 (the outer block)
        Ge, T, Kt = 32, 65536, 2880
        gen = torch.Generator("cpu").manual_seed(0)
        w = torch.exp(torch.randn(Ge, generator=gen))
        cnt = (w / w.sum() * T).floor().long() // 64 * 64
        cnt[-1] += T - int(cnt.sum())
        off = torch.zeros(Ge + 1, dtype=torch.int64)
        off[1:] = torch.cumsum(cnt, 0)
        xt = (torch.randn(T, Kt, generator=torch.Generator(dev).manual_seed(1), device=dev)).to(torch.bfloat16)
        offd = off.to(dev)
        kw = dict(mode="outer_block", outer_block_size=64, rowwise=True, columnwise=True)
        q = fq.quantize_grouped(xt, offd, **kw)
        ws = torch.empty(1 << 16, dtype=torch.uint8, device=dev)
        ms = _events_time(lambda i: fq.quantize_grouped(xt, offd, out=q, workspace=ws, **kw), iters, warmup)
        n = T * Kt
        nb = n * 2 + 2 * (n // 2) + 2 * (n // 16) + 2 * (n // 64) * 4
        return ("%d tokens x bf16[%d] in %d ragged expert groups (%d..%d rows), 1x64 outer, rowwise+columnwise" % (
            T, Kt, Ge, int(cnt.min()), int(cnt.max())), nb, ms, 2)

    def sr_ef_weight_qdq(iters, warmup, opts):
        g = torch.Generator(dev).manual_seed(0)
        Wt = torch.randn(8192, 8192, generator=g, device=dev) * 0.02
        r = torch.zeros_like(Wt)
        y = torch.empty(1, 8192, 8192, device=dev)
        ms = _events_time(lambda i: fq.qdq(Wt, stochastic=True, seed=0, step=i, residual=r, out_dtype=torch.float32,
                                           out=y), iters, warmup)
        return ("fp32[8192,8192] qdq, E4M3, SR + error feedback (x, r read; r, y written)", 4 * 8192 * 8192 * 4,
                ms, 1)

    return {
        "small_nvfp4_quantize": (small_nvfp4_quantize, 200, 10),
        "activations_outer_block": (_activations(dict(mode="outer_block", outer_block_size=64),
                                                 2 * codes + 2 * (M * K // 16) + 2 * (M * K // 64) * 4, 1), 200, 5),
        "activations_tensorwise": (activations_tensorwise, 200, 5),
        "activations_none": (_activations(dict(mode="none"), 2 * codes + 2 * (M * K // 16), 1), 200, 5),
        "activations_hadamard_outer_block": (_activations(dict(mode="outer_block", outer_block_size=64,
                                                               col_hadamard=True, hadamard_signs=0xA5C3),
                                                          2 * codes + 2 * (M * K // 16) + 2 * (M * K // 64) * 4, 1),
                                             200, 5),
        "activations_rowwise_outer_block": (_activations(dict(mode="outer_block", outer_block_size=64),
                                                         codes + M * K // 16 + (M * K // 64) * 4, 1,
                                                         columnwise=False), 200, 5),
        "activations_rowwise_sr": (_activations(dict(mode="none", stochastic=True), codes + M * K // 16, 1,
                                                columnwise=False), 200, 5),
        "dequantize_activations": (dequantize_activations, 200, 5),
        "moe_experts_e4m3": (_moe("e4m3"), 40, 3),
        "moe_experts_ue5m3": (_moe("ue5m3"), 40, 3),
        "moe_grouped_tokens": (moe_grouped_tokens, 80, 3),
        "mxfp4_project_mxfp8": (mxfp4_project_mxfp8, 200, 5),
        "sr_ef_weight_qdq": (sr_ef_weight_qdq, 20, 3),
    }


def extra_kernels(peak, only=None, iters=None, warmup=None, opts=None):
    """Time the other workloads; returns {name: record}."""
    import torch

    out = {}
    for name, (fn, it, wu) in _extra_workloads().items():
        if only and name != only:
            continue
        res = fn(iters or it, wu if warmup is None else warmup, opts or {})
        desc, nbytes, ms, launches = res[:4]
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"workload": desc, "bytes": nbytes, "us": round(ms * 1e3, 3), "GB/s": round(gbs, 1),
                     "frac_of_hbm": round(gbs / peak, 4), "launches": launches}
        if len(res) > 4:
            out[name]["parts"] = res[4]
        torch.cuda.empty_cache()
    return out


def run_ours(args, dist):
    import torch

    import block_scaled_fp4_quantize_gb300 as fq
    from block_scaled_fp4_quantize_gb300 import workloads as W

    fq.build()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    peak, peak_src = hbm_peak()

    x_host, _ = W.mxfp4_weight()
    xs = [x_host.to(dev) for _ in range(2)]          # 2 x (134 MB in + 134 MB out) > L2
    ys = [torch.empty_like(xs[0]) for _ in range(2)]

    def step(i):
        fq.mxfp4_fake_quantize(xs[i & 1], out=ys[i & 1])

    # the K timed steps as CUDA graph replays of the same calls (no Python
    # launch path between kernels); eager calls if capture is not possible
    sg = StepGraph(step, args.steps)
    sampler = ClockSampler(dev.index) if dist.rank == 0 else None
    t0 = time.time()
    # warm-up: at least W steps and at least 0.5 s of them, right before the
    # timed region, so that the clocks are at steady state when it starts
    _warm(step, args.warmup, min_seconds=0.5)
    dist.barrier()
    torch.cuda.synchronize()
    ms_region = sg.timed()  # synchronizes the device at its end
    dist.barrier()
    t1 = time.time()
    ms_total = dist.max(ms_region)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms_step = ms_total / args.steps
    value = MXFP4_BYTES * dist.world / (ms_step * 1e-3) / 1e9
    kernel_gbs = MXFP4_BYTES / (ms_step * 1e-3) / 1e9   # one launch per step: launch time == step time

    # end to end through the public API with HOST buffers: the library's
    # host entry point streams pinned host input -> device -> kernel -> pinned
    # host output in chunks, copies in both directions overlapping the kernel
    xh = x_host.pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    ws = torch.empty(fq.host_workspace_bytes(x_host.shape[-1]), dtype=torch.uint8, device=dev)

    def e2e_step(i):
        fq.mxfp4_fake_quantize_host(xh, out=yh, workspace=ws, device=dev, synchronize=False)

    e2e_ms = dist.max(_events_time(e2e_step, args.e2e_steps, 2, graph=False))
    torch.cuda.synchronize()
    link = link_calibration(xh, yh, dev)
    del xs, ys, ws

    extras = None
    if not args.no_extras and dist.rank == 0:
        extras = extra_kernels(peak)

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x_host, budget_s=12.0)

    if dist.rank != 0:
        return None
    line = {
        "metric": "FP4 quantize GB/s (bytes in+out) and % of GB300 HBM peak, 1 GPU",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / dist.world / B200_CUTE_DSL_GBS, 4),
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "mxfp4_weight: MXFP4 fake-quantize bf16[8192,8192] ~N(0,0.02), 0.1% edge blocks, "
                               "bf16 out", "shape": [8192, 8192], "bytes_per_step": MXFP4_BYTES,
                   "l2": "2 rotating input/output sets (537 MB > L2)", "parallelism": "replicas" if dist.world > 1 else "none",
                   "timing": ("CUDA events as the first and last nodes of the K steps' CUDA graphs" if sg.ok and sg.inside
                              else "CUDA events around K steps run as CUDA graph replays" if sg.ok
                              else "CUDA events around K eager steps"),
                   "warmup_policy": "at least W steps and 0.5 s of steps, no idle gap before the timed region"},
        "roofline": {"bound": "hbm", "achieved": round(kernel_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(kernel_gbs / peak, 4), "peak_source": peak_src,
                     "traffic": ncu_traffic("mxfp4_wide_kernel"), "kernel": "mxfp4_wide_kernel"},
        "e2e": {"value": round(MXFP4_BYTES / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": MXFP4_BYTES // 2, "d2h_bytes_per_step": MXFP4_BYTES // 2,
                "link": link, "frac_of_link": round(MXFP4_BYTES / (e2e_ms * 1e-3) / 1e9 / link["both_gbs"], 4)},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if extras is not None:
        line["kernels"] = extras
    return line


def link_calibration(xh, yh, dev, reps=5):
    """Host <-> device copy rates of the headline's pinned buffers on this
    box: host-to-device alone, device-to-host alone, and both at once on two
    streams (the overlap the end-to-end path relies on).  GB/s of bytes
    moved; the best of `reps`."""
    import torch

    nb = xh.numel() * xh.element_size()
    xd = torch.empty_like(xh, device=dev)
    yd = torch.empty_like(yh, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def best(fn, nbytes):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            a = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - a)
        return round(nbytes / min(ts) / 1e9, 1)

    def both():
        with torch.cuda.stream(s1):
            xd.copy_(xh, non_blocking=True)
        with torch.cuda.stream(s2):
            yh.copy_(yd, non_blocking=True)

    out = {"h2d_gbs": best(lambda: xd.copy_(xh, non_blocking=True), nb),
           "d2h_gbs": best(lambda: yh.copy_(yd, non_blocking=True), nb),
           "both_gbs": best(both, 2 * nb), "bytes_each_way": nb, "pinned": True}
    del xd, yd
    return out


# ---------------------------------------------------------------------------
# CPU oracle timings
# ---------------------------------------------------------------------------

def _oracle_rows_time(orc, xb, rows):
    t = time.perf_counter()
    orc.mxfp4_fake_quantize(xb[:rows])
    return time.perf_counter() - t


# The oracle on every host core: a process pool (started by spawn, so no
# state of this process, CUDA included, is inherited) whose workers each run
# the oracle, as it stands, on a contiguous slice of rows.  The input reaches
# them as a read-only memory map of one temporary .npy file (no shared-memory
# segment: its size is the host's choice); each worker keeps its output and
# returns a checksum.
_ORC = {}


def _orc_worker_init(path):
    import numpy as np

    import oracle as orc

    _ORC["orc"] = orc
    _ORC["x"] = np.load(path, mmap_mode="r")
    orc.mxfp4_fake_quantize(_ORC["x"][:1])  # load the library before the first timed task


def _orc_worker_rows(span):
    r0, r1 = span
    y = _ORC["orc"].mxfp4_fake_quantize(_ORC["x"][r0:r1])
    return int(y.view("u2").sum(dtype="u8"))


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class OraclePool:
    """`cores` oracle processes over one uint16 [rows, K] input; run(rows)
    times the leading `rows` rows split into one contiguous slice per
    process."""

    def __init__(self, xb, cores=None):
        import multiprocessing as mp
        import tempfile

        import numpy as np

        import oracle as orc

        orc.build()
        self.cores = cores or host_cores()
        self.dir = tempfile.mkdtemp(prefix="fp4q_oracle_")
        self.path = os.path.join(self.dir, "x.npy")
        np.save(self.path, np.ascontiguousarray(xb))
        self.pool = mp.get_context("spawn").Pool(self.cores, _orc_worker_init, (self.path,))

    def run(self, rows):
        """Seconds for the leading `rows` rows; the sum of the output's
        16-bit words is kept in self.checksum."""
        n = self.cores
        spans = [(rows * i // n, rows * (i + 1) // n) for i in range(n)]
        spans = [sp for sp in spans if sp[1] > sp[0]]
        t = time.perf_counter()
        sums = self.pool.map(_orc_worker_rows, spans, chunksize=1)
        dt = time.perf_counter() - t
        self.checksum = sum(sums)
        return dt

    def close(self):
        self.pool.close()
        self.pool.join()
        os.remove(self.path)
        os.rmdir(self.dir)


def cpu_baseline(x_host, budget_s=12.0):
    """The oracle, as it stands, on the host cores: every core (one process
    each, contiguous row slices of the whole headline tensor), beside the
    single-threaded figure on a bounded sample (leading rows)."""
    import numpy as np

    import oracle as orc

    orc.build()
    xb = x_host.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    t64 = _oracle_rows_time(orc, xb, 64)
    rows = int(max(64, min(xb.shape[0], 64 * budget_s / max(t64, 1e-6) / 4)))
    dt = _oracle_rows_time(orc, xb, rows)
    one = {"value": round(rows * xb.shape[1] * 4 / dt / 1e9, 4), "cores": 1,
           "sample": "leading %d of 8192 rows of the bf16[8192,8192] input (%.1f s)" % (rows, dt)}
    try:
        pool = OraclePool(xb)
        try:
            pool.run(xb.shape[0])  # warm-up pass
            reps, tot = 0, 0.0
            while reps < 3 or (tot < budget_s / 2 and reps < 50):
                tot += pool.run(xb.shape[0])
                reps += 1
        finally:
            pool.close()
    except Exception as e:  # no process pool on this host: the single-threaded figure alone
        return {"value": one["value"], "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": one["sample"],
                "all_cores": "unavailable: %s" % str(e).splitlines()[0][:200]}
    return {"value": round(xb.size * 4 * reps / tot / 1e9, 4), "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
            "sample": "the whole bf16[8192,8192] input, %d processes on contiguous row slices, %d passes (%.1f s)"
                      % (pool.cores, reps, tot),
            "single_core": one}


def run_reference(args, dist):
    """Reference arm: the CPU oracle on the host cores (one process per core,
    contiguous row slices), same metric and workload, each step the whole
    input; where no process pool can start, one core on a bounded sample
    (leading rows) per step."""
    if dist.rank != 0:
        return None
    import numpy as np
    import torch

    import oracle as orc
    from block_scaled_fp4_quantize_gb300 import workloads as W

    orc.build()
    x_host, _ = W.mxfp4_weight()
    xb = x_host.view(torch.int16).numpy().view(np.uint16)
    pool, note = None, None
    try:
        pool = OraclePool(xb)
        pool.run(xb.shape[0])
    except Exception as e:
        if pool is not None:
            pool.close()
        pool, note = None, "process pool unavailable: %s" % str(e).splitlines()[0][:200]
    try:
        if pool is not None:
            rows, cores = 8192, pool.cores
            step = lambda: pool.run(rows)
        else:
            t64 = _oracle_rows_time(orc, xb, 64)
            per_step_budget = 150.0 / max(1, args.steps + args.warmup)
            rows, cores = int(max(1, min(8192, 64 * per_step_budget / max(t64, 1e-6)))), 1
            step = lambda: _oracle_rows_time(orc, xb, rows)
        for _ in range(args.warmup):
            step()
        dt = sum(step() for _ in range(args.steps))
    finally:
        if pool is not None:
            pool.close()
    nbytes = rows * 8192 * 4 * args.steps
    value = nbytes / dt / 1e9
    sample = ("the whole input per step, %d processes on contiguous row slices" % cores if rows == 8192 and cores > 1
              else "leading %d of 8192 rows per step" % rows)
    cpu = {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    if note:
        cpu["all_cores"] = note
    return {
        "impl": "reference",
        "metric": "FP4 quantize GB/s (bytes in+out) and % of GB300 HBM peak, 1 GPU",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "mxfp4_weight: MXFP4 fake-quantize bf16[8192,8192] ~N(0,0.02), 0.1% edge blocks, "
                               "bf16 out", "shape": [8192, 8192], "sample_rows_per_step": rows},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        # rank 0 alone times the oracle; the other ranks exit without work
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        ref = argparse.Namespace(rank=0, world=int(os.environ.get("WORLD_SIZE", "1")), local=0)
        print(json.dumps(run_reference(args, ref)))
        return 0
    if args.only:
        import block_scaled_fp4_quantize_gb300 as fq

        fq.build()
        peak, _ = hbm_peak()
        rec = extra_kernels(peak, only=args.only, iters=args.steps, warmup=args.warmup,
                            opts={"experts": args.experts})
        if not rec:
            raise SystemExit("unknown workload %r" % args.only)
        print(json.dumps({"only": args.only, **rec[args.only]}))
        return 0
    dist = Dist()
    try:
        line = run_ours(args, dist)
    finally:
        dist.close()
    if line is not None:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
