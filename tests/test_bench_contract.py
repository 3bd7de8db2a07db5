"""bench.py's reference arm (the oracle timed on the host cores) prints one
JSON line with the keys of the benchmark line, and under a multi-rank launch
only rank 0 prints it."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _run(extra_env=None):
    env = dict(os.environ, **(extra_env or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)


def test_reference_arm_prints_one_line_with_the_contract_keys():
    out = _run()
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert KEYS <= set(rec)
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["higher_is_better"] is True
    assert rec["value"] > 0 and rec["steps"] == 1 and rec["warmup"] == 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    assert rec["config"]["workload"].startswith("mxfp4_weight")


def test_reference_arm_other_ranks_exit_quietly():
    out = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_oracle_pool_matches_one_process():
    """The all-cores CPU baseline runs the oracle unchanged on row slices:
    the slices' outputs add up to the output of one call on every row."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from block_scaled_fp4_quantize_gb300 import workloads as W

    x = W.lognormal((96, 256), 61, sigma=3.0).view(__import__("torch").int16).numpy().view(np.uint16)
    pool = bench.OraclePool(x, cores=3)
    try:
        pool.run(96)
        got = pool.checksum
        pool.run(50)  # a leading part, uneven slices
        part = pool.checksum
    finally:
        pool.close()
    assert got == int(oracle.mxfp4_fake_quantize(x).view("u2").sum(dtype="u8"))
    assert part == int(oracle.mxfp4_fake_quantize(x[:50]).view("u2").sum(dtype="u8"))


def test_graph_split_covers_every_call_once():
    """The timed calls are split into a head graph (holding the start event),
    replays of a body graph and a tail graph (holding the end event): the
    parts add up to n, the tail is 1 .. chunk calls when n > chunk, and a
    single graph holds both events otherwise."""
    sys.path.insert(0, ROOT)
    import bench

    for n in list(range(1, 420)) + [25000]:
        for chunk in (1, 7, 100):
            h, nb, ch, t = bench.graph_split(n, chunk)
            assert h + nb * ch + t == n
            assert h == min(n, chunk) and ch == min(n, chunk)
            assert (t == 0) == (n <= chunk)
            assert t == 0 or 1 <= t <= chunk
