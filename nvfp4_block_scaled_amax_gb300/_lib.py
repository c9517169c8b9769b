"""ctypes loader for libnvfp4.so (the C ABI of include/nvfp4.h).

Argument marshalling only: every step of the quantize path runs in the
library's CUDA kernels.  There is no fallback: if the library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnvfp4.so")

NVFP4_OK = 0
STATUS_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_DTYPE", 5: "ERR_FLAGS",
                6: "ERR_CUDA", 7: "ERR_TIMEOUT"}

# Every symbol the header declares.
EXPORTS = ("nvfp4_status_string", "nvfp4_scale_bytes", "nvfp4_compute_amax", "nvfp4_compute_amax_rht",
           "nvfp4_quantize_1d", "nvfp4_quantize_2d", "nvfp4_quantize_row_scaled", "nvfp4_quantize_rht",
           "nvfp4_quantize_1d_single_pass", "nvfp4_quantize_2d_single_pass", "nvfp4_quantize_rht_single_pass",
           "nvfp4_quantize_2d_single_pass_noalloc", "nvfp4_quantize_grouped_1d", "nvfp4_quantize_grouped_2d",
           "nvfp4_quantize_grouped_1d_single_pass", "nvfp4_quantize_grouped_2d_single_pass",
           "nvfp4_quantize_1d_sr", "nvfp4_quantize_2d_sr",
           "nvfp4_dequantize", "nvfp4_swizzle_scales", "nvfp4_device_status")
SINGLE_PASS_WORKSPACE_BYTES = 4096
MAX_GROUPS = 64


class Output(ctypes.Structure):
    """nvfp4_output."""
    _fields_ = [("data_row", ctypes.c_void_p), ("scale_row", ctypes.c_void_p), ("amax_row", ctypes.c_void_p),
                ("data_col", ctypes.c_void_p), ("scale_col", ctypes.c_void_p), ("amax_col", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -m nvfp4_block_scaled_amax_gb300.build` "
                "(nvcc, sm_103a); there is no non-CUDA implementation")
        L = ctypes.CDLL(p)
        i64, vp, u32, c_int, uint = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint
        L.nvfp4_status_string.argtypes = [c_int]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_scale_bytes.argtypes = [i64, i64, uint, ctypes.POINTER(ctypes.c_size_t)]
        L.nvfp4_compute_amax.argtypes = [vp, c_int, i64, i64, vp, vp, vp, vp]
        L.nvfp4_compute_amax_rht.argtypes = [vp, c_int, i64, i64, u32, vp, vp, vp, vp]
        for name in ("nvfp4_quantize_1d", "nvfp4_quantize_2d", "nvfp4_quantize_row_scaled"):
            getattr(L, name).argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, vp, vp]
        L.nvfp4_quantize_rht.argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, u32, vp, vp]
        for name in ("nvfp4_quantize_1d_single_pass", "nvfp4_quantize_2d_single_pass"):
            getattr(L, name).argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, vp, vp, vp]
        L.nvfp4_quantize_rht_single_pass.argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, u32, vp, vp,
                                                     vp]
        L.nvfp4_quantize_2d_single_pass_noalloc.argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, vp,
                                                           vp]
        for name in ("nvfp4_quantize_1d_sr", "nvfp4_quantize_2d_sr"):
            getattr(L, name).argtypes = [vp, c_int, i64, i64, ctypes.POINTER(Output), uint, vp, vp, vp]
        for name in ("nvfp4_quantize_grouped_1d", "nvfp4_quantize_grouped_2d"):
            getattr(L, name).argtypes = [vp, c_int, i64, c_int, ctypes.POINTER(i64), ctypes.POINTER(Output), uint,
                                         vp, vp]
        for name in ("nvfp4_quantize_grouped_1d_single_pass", "nvfp4_quantize_grouped_2d_single_pass"):
            getattr(L, name).argtypes = [vp, c_int, i64, c_int, ctypes.POINTER(i64), ctypes.POINTER(Output), uint,
                                         vp, vp, vp]
        L.nvfp4_dequantize.argtypes = [vp, vp, vp, i64, i64, uint, vp, c_int, vp]
        L.nvfp4_swizzle_scales.argtypes = [vp, vp, i64, i64, vp]
        L.nvfp4_device_status.argtypes = [ctypes.POINTER(u32), c_int]
        for name in EXPORTS[1:]:
            getattr(L, name).restype = c_int
        if path is None:
            _lib = L
        return L


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = load().nvfp4_status_string(status).decode()
        super().__init__(f"{what}: {msg}")


def check(status: int, what: str) -> None:
    if status != NVFP4_OK:
        raise NVFP4Error(status, what)
