"""fp4_quantize_noalloc: the quantize entry point for callers that cannot
allocate device memory (a pool owns the whole device, or an allocation may
not block).  Its scratch is a static device array shared by all calls, so
this test makes two calls in a row -- the second on data with a smaller
amplitude, which would expose a stale amax left in the shared array -- and
compares both with fp4_quantize given a freshly allocated workspace."""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp4_quantize_gb300 import _capi
from block_scaled_fp4_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(lib, x, noalloc, mode="tensorwise", ob=0):
    G, M, K = 1, x.shape[0], x.shape[1]
    p = _capi.new_params(lib)
    p.G, p.M, p.K, p.ld = G, M, K, K
    p.mode = {"tensorwise": _capi.MODE_TENSORWISE, "outer_block": _capi.MODE_OUTER_BLOCK}[mode]
    p.outer_block_size, p.out_mask = ob, 3
    bufs = {
        "row_codes": torch.empty(M * K // 2, dtype=torch.uint8, device="cuda"),
        "row_scales": torch.empty(M * K // 16, dtype=torch.uint8, device="cuda"),
        "col_codes": torch.empty(M * K // 2, dtype=torch.uint8, device="cuda"),
        "col_scales": torch.empty(M * K // 16, dtype=torch.uint8, device="cuda"),
        "row_outer": torch.empty(max(1, M * K // max(ob, 1)), dtype=torch.float32, device="cuda"),
        "col_outer": torch.empty(max(1, M * K // max(ob, 1)), dtype=torch.float32, device="cuda"),
        "tile_outer": torch.empty(1, dtype=torch.float32, device="cuda"),
    }
    names = ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer")
    out = _capi.Outputs(*[ctypes.c_void_p(bufs[n].data_ptr()) for n in names])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    xp = ctypes.c_void_p(x.data_ptr())
    if noalloc:
        rc = lib.fp4_quantize_noalloc(ctypes.byref(p), xp, ctypes.byref(out), None, stream)
    else:
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        rc = lib.fp4_quantize(ctypes.byref(p), xp, ctypes.byref(out), None, ctypes.c_void_p(ws.data_ptr()), 256,
                              stream)
    assert rc == 0, _capi.STATUS.get(rc)
    torch.cuda.synchronize()
    keep = names if mode == "outer_block" else ("row_codes", "row_scales", "col_codes", "col_scales", "tile_outer")
    return {n: bufs[n].cpu().numpy() for n in keep}


def test_noalloc_matches_fp4_quantize_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _capi.load()
    big = W.activations(M=256, K=576, n_cols=3, n_rows=1).cuda()       # large amax first
    small = (W.lognormal((256, 576), 31, sigma=0.5) * 0.01).cuda()     # then a much smaller one
    for x in (big, small):
        a = _run(lib, x, noalloc=True)
        b = _run(lib, x, noalloc=False)
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    # modes that need no scratch pass straight through
    a = _run(lib, big, noalloc=True, mode="outer_block", ob=64)
    b = _run(lib, big, noalloc=False, mode="outer_block", ob=64)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_noalloc_rejects_bad_parameters_like_fp4_quantize():
    lib = _capi.load()
    p = _capi.new_params(lib)
    p.M, p.K, p.ld = 64, 72, 72  # K % 16 != 0
    out = _capi.Outputs()
    assert lib.fp4_quantize_noalloc(ctypes.byref(p), None, ctypes.byref(out), None, None) == -3
    assert lib.fp4_quantize_noalloc(None, None, ctypes.byref(out), None, None) == -1
