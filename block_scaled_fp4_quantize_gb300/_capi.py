"""ctypes declarations of the C ABI in ``include/fp4q.h`` (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

from . import _builder as _build

FP4Q_OK = 0
STATUS = {
    0: "FP4Q_OK", -1: "FP4Q_ERR_NULL", -2: "FP4Q_ERR_DTYPE", -3: "FP4Q_ERR_SHAPE", -4: "FP4Q_ERR_MODE",
    -5: "FP4Q_ERR_UNSUPPORTED", -6: "FP4Q_ERR_WORKSPACE", -7: "FP4Q_ERR_CUDA", -8: "FP4Q_ERR_ABI",
    -9: "FP4Q_ERR_ALIGN", -10: "FP4Q_ERR_TIMEOUT",
}
BF16, FP32, FP16 = 1, 2, 3
MODE_NONE, MODE_TENSORWISE, MODE_OUTER_BLOCK = 0, 1, 2
SCALE_E4M3, SCALE_UE5M3 = 0, 1
SCALE_LAYOUT_LINEAR, SCALE_LAYOUT_MMA = 0, 1
ABI_VERSION = 4  # FP4Q_ABI_VERSION of include/fp4q.h
RNE, STOCHASTIC = 0, 1
OUT_ROW, OUT_COL = 1, 2

# every symbol include/fp4q.h declares
EXPORTS = ("fp4q_params_init", "fp4q_query_sizes", "fp4_quantize", "fp4_dequantize", "fp4_qdq",
           "mxfp4_fake_quantize", "mxfp4_fake_quantize_host", "mxfp4_project_mxfp8", "fp4_tensor_amax", "fp4_quantize_grouped",
           "fp4q_query_sizes_grouped", "fp4q_status_string",
           "fp4q_abi_version", "fp4_quantize_noalloc", "fp4q_device_status", "fp4q_set_device_timeout_flag")


class Params(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32), ("out_mask", ctypes.c_uint32),
        ("G", ctypes.c_int64), ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("ld", ctypes.c_int64),
        ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("mode", ctypes.c_int32),
        ("outer_block_size", ctypes.c_int32), ("outer_2d", ctypes.c_int32), ("inner_2d", ctypes.c_int32),
        ("scale_format", ctypes.c_int32), ("rounding", ctypes.c_int32),
        ("seed", ctypes.c_uint64), ("step", ctypes.c_uint32), ("use_precomputed_outer", ctypes.c_int32),
        ("scale_layout", ctypes.c_int32), ("col_hadamard", ctypes.c_int32), ("hadamard_signs", ctypes.c_uint32),
        ("precomputed_amax", ctypes.c_int32),
        ("sr_global_rows", ctypes.c_int64), ("sr_row_offset", ctypes.c_int64), ("sr_matrix_offset", ctypes.c_int64),
    ]


class Outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer")]


class Sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("row_codes", "row_scales", "row_outer", "col_codes", "col_scales", "col_outer", "tile_outer",
                 "workspace")]


class FP4QError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__("%s%s (%d)" % (where + ": " if where else "", STATUS.get(status, "unknown status"), status))


_libs = {}


def load(fast_math: bool = False, path: str | None = None):
    """Load the shared library (building it first if it is missing or stale).

    There is no fallback: if the library cannot be built or loaded this raises."""
    key = path or ("fm" if fast_math else "std")
    if key in _libs:
        return _libs[key]
    if path is None:
        path = _build.lib_path(fast_math)
        if not os.path.exists(path) or os.environ.get("FP4Q_AUTOBUILD", "1") == "1":
            path = _build.build(fast_math=fast_math)
    L = ctypes.CDLL(path)
    P, I, PP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(Params)
    L.fp4q_params_init.restype = None
    L.fp4q_params_init.argtypes = [PP]
    L.fp4q_query_sizes.restype = I
    L.fp4q_query_sizes.argtypes = [PP, ctypes.POINTER(Sizes)]
    L.fp4_quantize.restype = I
    L.fp4_quantize.argtypes = [PP, P, ctypes.POINTER(Outputs), P, P, ctypes.c_size_t, P]
    L.fp4_dequantize.restype = I
    L.fp4_dequantize.argtypes = [PP, I, P, P, P, P, P]
    L.fp4_qdq.restype = I
    L.fp4_qdq.argtypes = [PP, I, P, P, P, P, P, ctypes.c_size_t, P]
    L.mxfp4_fake_quantize.restype = I
    L.mxfp4_fake_quantize.argtypes = [PP, P, P, P]
    L.mxfp4_fake_quantize_host.restype = I
    L.mxfp4_fake_quantize_host.argtypes = [PP, P, P, P, ctypes.c_size_t, P]
    L.mxfp4_project_mxfp8.restype = I
    L.mxfp4_project_mxfp8.argtypes = [PP, P, P, P, P, P, P, P]
    L.fp4_quantize_grouped.restype = I
    L.fp4_quantize_grouped.argtypes = [PP, P, P, ctypes.c_int64, ctypes.POINTER(Outputs), P, ctypes.c_size_t, P]
    L.fp4q_query_sizes_grouped.restype = I
    L.fp4q_query_sizes_grouped.argtypes = [PP, ctypes.c_int64, ctypes.POINTER(Sizes)]
    L.fp4_tensor_amax.restype = I
    L.fp4_tensor_amax.argtypes = [PP, P, P, P, P]
    L.fp4_quantize_noalloc.restype = I
    L.fp4_quantize_noalloc.argtypes = [PP, P, ctypes.POINTER(Outputs), P, P]
    L.fp4q_status_string.restype = ctypes.c_char_p
    L.fp4q_status_string.argtypes = [I]
    L.fp4q_abi_version.restype = I
    L.fp4q_abi_version.argtypes = []
    L.fp4q_device_status.restype = I
    L.fp4q_device_status.argtypes = [I, P]
    L.fp4q_set_device_timeout_flag.restype = I
    L.fp4q_set_device_timeout_flag.argtypes = []
    if L.fp4q_abi_version() != ABI_VERSION:
        raise RuntimeError("libfp4q ABI version mismatch")
    _libs[key] = L
    return L


def new_params(lib=None) -> Params:
    p = Params()
    (lib or load()).fp4q_params_init(ctypes.byref(p))
    return p


def check(status: int, where: str = ""):
    if status != FP4Q_OK:
        raise FP4QError(status, where)
