"""CPU oracle for NVFP4 quantize-with-transpose (test infrastructure only).

This package wraps ``nvfp4_oracle.c``: a plain, single-threaded C restatement
of what the quantize path computes (see the header of that file for every
step, its source passage and the readings taken where the pages are silent).
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the library itself never does, and this package
imports nothing from the library.

Arrays are numpy.  BF16 tensors travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP32 = 1
MODE_1D = 0
MODE_2D = 1
MODE_RHT = 2
MODE_ROW_SCALED = 3
MODES = {"1d": MODE_1D, "2d": MODE_2D, "rht": MODE_RHT, "row_scaled": MODE_ROW_SCALED}

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (no SIMD intrinsics, no FMA contraction).

    ``NVFP4_ORACLE_LIB`` names an already built copy to load instead; the
    planted-mistake tests use it to run the pins against altered copies."""
    override = os.environ.get("NVFP4_ORACLE_LIB")
    if override:
        return override
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, u8p, f32p, vp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_bf16_rn.argtypes = [ctypes.c_float]
            L.oracle_f32_to_bf16_rn.restype = ctypes.c_uint16
            L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            L.oracle_e2m1_value.restype = ctypes.c_float
            L.oracle_e2m1_rn_satfinite.argtypes = [ctypes.c_float]
            L.oracle_e2m1_rn_satfinite.restype = ctypes.c_uint8
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_rn_satfinite.argtypes = [ctypes.c_float]
            L.oracle_e4m3_rn_satfinite.restype = ctypes.c_uint8
            L.oracle_global_encode_scale.argtypes = [ctypes.c_float]
            L.oracle_global_encode_scale.restype = ctypes.c_float
            L.oracle_block_scale.argtypes = [ctypes.c_float, ctypes.c_float]
            L.oracle_block_scale.restype = ctypes.c_uint8
            L.oracle_encode_factor.argtypes = [ctypes.c_uint8, ctypes.c_float]
            L.oracle_encode_factor.restype = ctypes.c_float
            L.oracle_amax.argtypes = [vp, ctypes.c_int, i64]
            L.oracle_amax.restype = ctypes.c_float
            L.oracle_rht_amax.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_uint32]
            L.oracle_rht_amax.restype = ctypes.c_float
            L.oracle_hadamard16.argtypes = [ctypes.c_int, ctypes.c_int]
            L.oracle_hadamard16.restype = ctypes.c_int
            L.oracle_rht16.argtypes = [f32p, ctypes.c_uint32, ctypes.c_int, f32p]
            L.oracle_rht16.restype = None
            L.oracle_rht_columns.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_uint32, ctypes.c_int, vp, i64,
                                             f32p]
            L.oracle_rht_columns.restype = ctypes.c_int
            L.oracle_quantize.argtypes = [
                ctypes.c_int, vp, ctypes.c_int, i64, i64,
                ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_uint32,
                vp, i64, vp, i64,
                u8p, u8p, f32p, u8p, u8p, f32p]
            L.oracle_quantize.restype = ctypes.c_int
            L.oracle_quantize_sr.argtypes = [
                ctypes.c_int, vp, ctypes.c_int, i64, i64,
                ctypes.c_int, ctypes.c_float, ctypes.c_float, vp,
                vp, i64, vp, i64,
                u8p, u8p, f32p, u8p, u8p, f32p]
            L.oracle_quantize_sr.restype = ctypes.c_int
            L.oracle_e2m1_sr_satfinite.argtypes = [ctypes.c_float, ctypes.c_uint8]
            L.oracle_e2m1_sr_satfinite.restype = ctypes.c_uint8
            L.oracle_e2m1_sr_array.argtypes = [vp, vp, vp, i64]
            L.oracle_e2m1_sr_array.restype = None
            L.oracle_swizzle_offset.argtypes = [i64, i64, i64]
            L.oracle_swizzle_offset.restype = i64
            L.oracle_swizzle_scales.argtypes = [u8p, u8p, i64, i64]
            L.oracle_swizzle_scales.restype = ctypes.c_int
            L.oracle_dequantize.argtypes = [u8p, u8p, f32p, ctypes.c_int, i64, i64, ctypes.c_int, vp]
            L.oracle_dequantize.restype = ctypes.c_int
            for name in ("oracle_e2m1_array", "oracle_e4m3_array", "oracle_bf16_array"):
                getattr(L, name).argtypes = [vp, vp, i64]
                getattr(L, name).restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return FP32
    raise TypeError("oracle input must be uint16 (BF16 bits) or float32")


# ---------------------------------------------------------------------------
# Scalar helpers (used by the pins)
# ---------------------------------------------------------------------------

def e2m1(v: float) -> int:
    return int(lib().oracle_e2m1_rn_satfinite(float(v)))


def e2m1_sr(v: float, rb: int) -> int:
    """Stochastically rounded E2M1 code of v with random byte rb."""
    return int(lib().oracle_e2m1_sr_satfinite(float(v), int(rb) & 0xFF))


def e2m1_sr_array(v: np.ndarray, rb: np.ndarray) -> np.ndarray:
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    r = np.ascontiguousarray(np.broadcast_to(rb, np.shape(v)), dtype=np.uint8).ravel()
    out = np.empty(flat.size, dtype=np.uint8)
    lib().oracle_e2m1_sr_array(_ptr(flat), _ptr(r), _ptr(out), flat.size)
    return out.reshape(np.shape(v))


def e2m1_value(code: int) -> float:
    return float(lib().oracle_e2m1_value(code))


def e4m3(v: float) -> int:
    return int(lib().oracle_e4m3_rn_satfinite(float(v)))


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(code))


def bf16_round(v: float) -> int:
    return int(lib().oracle_f32_to_bf16_rn(float(v)))


def global_encode_scale(amax: float) -> float:
    return float(lib().oracle_global_encode_scale(float(amax)))


def block_scale(block_amax: float, g: float) -> int:
    return int(lib().oracle_block_scale(float(block_amax), float(g)))


def encode_factor(s: int, g: float) -> float:
    return float(lib().oracle_encode_factor(s, float(g)))


def hadamard16() -> np.ndarray:
    L = lib()
    return np.array([[L.oracle_hadamard16(o, i) for i in range(16)] for o in range(16)], dtype=np.int64)


def rht16(v: np.ndarray, mask: int, round_bf16: bool) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (16,)
    t = np.empty(16, dtype=np.float32)
    lib().oracle_rht16(_ptr(v), mask & 0xFFFF, int(round_bf16), _ptr(t))
    return t


def rht_columns(x: np.ndarray, mask: int, round_bf16: bool, cols: np.ndarray | None = None) -> np.ndarray:
    """The column-block RHT of the columns ``cols`` of x (all when None), as
    a [len(cols), M] float32 array (row k = column cols[k] of x transformed):
    rounded to BF16 like the column-wise quantize reads them, or the FP32 sums
    before that rounding (round_bf16=False)."""
    x = np.ascontiguousarray(x)
    M, N = x.shape
    ids = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nc = N if ids is None else ids.size
    out = np.empty((nc, M), dtype=np.float32)
    rc = lib().oracle_rht_columns(_ptr(x), _dtype_code(x), M, N, mask & 0xFFFF, int(round_bf16), _ptr(ids),
                                  0 if ids is None else ids.size, _ptr(out))
    if rc != 0:
        raise ValueError("RHT columns need M % 16 == 0")
    return out


def encode_array(v: np.ndarray, fmt: str) -> np.ndarray:
    """Element-wise E2M1 / E4M3 / BF16 encoding of a float32 array."""
    L = lib()
    fn = {"e2m1": L.oracle_e2m1_array, "e4m3": L.oracle_e4m3_array, "bf16": L.oracle_bf16_array}[fmt]
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(flat.size, dtype=np.uint16 if fmt == "bf16" else np.uint8)
    fn(_ptr(flat), _ptr(out), flat.size)
    return out.reshape(np.shape(v))


# ---------------------------------------------------------------------------
# Matrix operations
# ---------------------------------------------------------------------------

def amax(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x)
    return float(lib().oracle_amax(_ptr(x), _dtype_code(x), x.size))


def rht_amax(x: np.ndarray, mask: int) -> float:
    x = np.ascontiguousarray(x)
    M, N = x.shape
    return float(lib().oracle_rht_amax(_ptr(x), _dtype_code(x), M, N, mask & 0xFFFF))


def quantize(mode: str, x: np.ndarray, rowwise: bool = True, colwise: bool = True,
             sign_mask: int = 0, amax: tuple[float, float] | None = None,
             rows: np.ndarray | None = None, cols: np.ndarray | None = None,
             rbits: np.ndarray | None = None) -> dict:
    """NVFP4-quantizes x (M x N; uint16 BF16 bits or float32).

    Returns compact outputs: ``row_data`` [nr, N/2], ``row_scale`` [nr, N/16],
    ``amax_row`` (1 value, or nr for row-scaled), ``col_data`` [nc, M/2],
    ``col_scale`` [nc, M/16], ``amax_col``.  ``rows`` / ``cols`` select which
    rows of the row-wise output and which columns of x (rows of the
    column-wise output) to produce; None means all.  ``amax`` = (row, col)
    uses a given amax pair instead of reducing x.  ``rbits`` (uint8, the
    shape of x): stochastic rounding of the codes, modes 1d and 2d, element
    (y, j) using rbits[y, j] in both outputs.
    """
    x = np.ascontiguousarray(x)
    M, N = x.shape
    m = MODES[mode]
    row_ids = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    col_ids = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = 0 if not rowwise else (M if row_ids is None else row_ids.size)
    nc = 0 if not colwise else (N if col_ids is None else col_ids.size)
    n_row_arg = 0 if not rowwise else (-1 if row_ids is None else row_ids.size)
    n_col_arg = 0 if not colwise else (-1 if col_ids is None else col_ids.size)
    row_data = np.zeros((nr, N // 2), dtype=np.uint8)
    row_scale = np.zeros((nr, N // 16), dtype=np.uint8)
    col_data = np.zeros((nc, M // 2), dtype=np.uint8)
    col_scale = np.zeros((nc, M // 16), dtype=np.uint8)
    amax_row = np.zeros(max(nr, 1) if m == MODE_ROW_SCALED else 1, dtype=np.float32)
    amax_col = np.zeros(1, dtype=np.float32)
    given = amax is not None
    ar, ac = (amax if given else (0.0, 0.0))
    if rbits is None:
        rc = lib().oracle_quantize(
            m, _ptr(x), _dtype_code(x), M, N, int(given), float(ar), float(ac), sign_mask & 0xFFFF,
            _ptr(row_ids), n_row_arg, _ptr(col_ids), n_col_arg,
            _ptr(row_data), _ptr(row_scale), _ptr(amax_row),
            _ptr(col_data), _ptr(col_scale), _ptr(amax_col))
    else:
        rb = np.ascontiguousarray(rbits, dtype=np.uint8)
        if rb.shape != (M, N):
            raise ValueError("rbits must hold one byte per element of x")
        rc = lib().oracle_quantize_sr(
            m, _ptr(x), _dtype_code(x), M, N, int(given), float(ar), float(ac), _ptr(rb),
            _ptr(row_ids), n_row_arg, _ptr(col_ids), n_col_arg,
            _ptr(row_data), _ptr(row_scale), _ptr(amax_row),
            _ptr(col_data), _ptr(col_scale), _ptr(amax_col))
    if rc != 0:
        raise ValueError(f"oracle: shape {M}x{N} not defined for mode {mode}")
    return {"row_data": row_data, "row_scale": row_scale, "amax_row": amax_row[:max(nr, 1)],
            "col_data": col_data, "col_scale": col_scale, "amax_col": amax_col}


def quantize_grouped(mode: str, x: np.ndarray, splits, rowwise: bool = True, colwise: bool = True) -> list[dict]:
    """Grouped (multi-tensor) quantize: x stacks G tensors along its first
    dimension, tensor g being rows [sum(splits[:g]), sum(splits[:g+1])) with
    the common last dimension N.  Each member is quantized as a tensor of its
    own: its own amax (so its own global scale), block scales and codes, and
    its column-wise output is the transpose of its own rows only.

    Reading of "Implement row-scaled NVFP4 fprop recipe" (Important Files
    Changed, grouped_tensor_storage.py): a grouped tensor keeps its members'
    amaxes side by side and slices them per member tensor, so every member
    carries its own amax.  Modes 1d and 2d (row-scaled needs no grouping: each
    row is already a tensor of its own).  Returns one ``quantize`` result per
    member, in order.
    """
    x = np.ascontiguousarray(x)
    if mode not in ("1d", "2d"):
        raise ValueError("grouped quantize: modes 1d and 2d")
    splits = [int(m) for m in splits]
    if any(m < 0 for m in splits) or sum(splits) != x.shape[0]:
        raise ValueError("grouped quantize: splits must be non-negative and sum to the rows of x")
    out, r = [], 0
    for m in splits:
        out.append(quantize(mode, x[r:r + m], rowwise=rowwise, colwise=colwise))
        r += m
    return out


def swizzle_offset(r: int, c: int, C: int) -> int:
    return int(lib().oracle_swizzle_offset(r, c, C))


def swizzle(compact: np.ndarray) -> np.ndarray:
    compact = np.ascontiguousarray(compact, dtype=np.uint8)
    R, C = compact.shape
    out = np.zeros(R * C, dtype=np.uint8)
    if lib().oracle_swizzle_scales(_ptr(compact), _ptr(out), R, C) != 0:
        raise ValueError("swizzled layout needs rows % 128 == 0 and scale cols % 4 == 0")
    return out


def dequantize(data: np.ndarray, scale: np.ndarray, amax: np.ndarray, per_row: bool,
               out_dtype: str = "bf16") -> np.ndarray:
    """Dequantizes packed codes with compact scales; returns uint16 BF16 bits or float32."""
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    amax = np.ascontiguousarray(amax, dtype=np.float32)
    rows, half = data.shape
    cols = half * 2
    od = BF16 if out_dtype == "bf16" else FP32
    out = np.empty((rows, cols), dtype=np.uint16 if od == BF16 else np.float32)
    rc = lib().oracle_dequantize(_ptr(data), _ptr(scale), _ptr(amax), int(per_row), rows, cols, od, _ptr(out))
    if rc != 0:
        raise ValueError("oracle dequantize: bad shape")
    return out
