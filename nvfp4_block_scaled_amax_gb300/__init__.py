"""NVFP4 quantize-with-transpose on one GB300 GPU (sm_103a).

A thin PyTorch-facing binding of ``libnvfp4.so`` (C ABI in include/nvfp4.h).
PyTorch supplies device memory and the current CUDA stream; every step of the
computation (amax, scales, codes, transposition, swizzled scale layout,
Hadamard transform, dequantize) runs in the library's CUDA kernels.

    q = quantize(x, mode="2d", swizzled=True)    # amax + fused cast, one launch
    xr = dequantize(q.data_row, q.scale_row, q.amax_row, swizzled=True)

Modes: "1d" (1x16 blocks), "2d" (16x16 tiles), "rht" (random Hadamard
transform on the column-wise path) and "row_scaled" (one amax per row,
row-wise only).  ``quantize_grouped`` quantizes several tensors stacked along
the first dimension, each with its own amax (one launch for bfloat16);
``quantize_sr`` rounds the codes stochastically with caller-supplied random
bytes.

Paths for "1d" / "2d" / "rht": "single_pass" (one persistent kernel: amax,
grid barrier, cast; x read from HBM once; needs a small workspace, which
this module keeps per device and stream) and "two_pass" (an amax kernel,
then the cast kernel; needed for skip_amax).  "auto" picks single_pass for
1d / 2d when it applies and two_pass for rht (measured faster there).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import NVFP4Error

ROWWISE = 1
COLWISE = 2
SWIZZLED = 4
SKIP_AMAX = 8
ROW_SCALED = 16
BF16 = 0
FP32 = 1

__all__ = ["NVFP4Tensor", "NVFP4Error", "empty", "compute_amax", "compute_amax_rht", "quantize", "QuantizePlan",
           "single_pass_workspace", "reset_workspaces",
           "quantize_1d", "quantize_2d", "quantize_rht", "quantize_row_scaled", "quantize_grouped", "quantize_sr",
           "dequantize",
           "swizzle_scales", "scale_bytes", "device_status"]


@dataclass
class NVFP4Tensor:
    """Row-wise and/or column-wise NVFP4 data of an M x N tensor.

    data_row [M, N/2] uint8, scale_row [M*N/16] uint8, amax_row [1] (row-scaled: [M]) float32;
    data_col [N, M/2] uint8, scale_col [N*M/16] uint8, amax_col [1] float32.
    Scale buffers are flat: compact [rows][cols/16] or the cuBLAS 128x4 layout.
    """
    M: int
    N: int
    data_row: torch.Tensor | None = None
    scale_row: torch.Tensor | None = None
    amax_row: torch.Tensor | None = None
    data_col: torch.Tensor | None = None
    scale_col: torch.Tensor | None = None
    amax_col: torch.Tensor | None = None
    swizzled: bool = False
    row_scaled: bool = False

    def c_struct(self) -> _lib.Output:
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        return _lib.Output(p(self.data_row), p(self.scale_row), p(self.amax_row),
                           p(self.data_col), p(self.scale_col), p(self.amax_col))


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return BF16
    if x.dtype == torch.float32:
        return FP32
    raise TypeError(f"NVFP4 quantize takes bfloat16 or float32 input, got {x.dtype}")


def _require_cuda(*ts: torch.Tensor | None) -> None:
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors passed to libnvfp4 must be contiguous CUDA tensors")


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class _OnDevice:
    """Makes `device` current for the library call (a no-op when it already is)."""
    __slots__ = ("idx", "prev")

    def __init__(self, device: torch.device):
        self.idx = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def empty(M: int, N: int, rowwise: bool = True, colwise: bool = True, row_scaled: bool = False,
          swizzled: bool = False, device: torch.device | str = "cuda") -> NVFP4Tensor:
    """Allocates (with PyTorch) the output buffers of an M x N quantization."""
    dev = torch.device(device)
    q = NVFP4Tensor(M, N, swizzled=swizzled, row_scaled=row_scaled)
    if rowwise:
        q.data_row = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
        q.scale_row = torch.empty(M * (N // 16), dtype=torch.uint8, device=dev)
        q.amax_row = torch.empty(M if row_scaled else 1, dtype=torch.float32, device=dev)
    if colwise:
        q.data_col = torch.empty((N, M // 2), dtype=torch.uint8, device=dev)
        q.scale_col = torch.empty(N * (M // 16), dtype=torch.uint8, device=dev)
        q.amax_col = torch.empty(1, dtype=torch.float32, device=dev)
    return q


_workspaces: dict = {}


def single_pass_workspace(device: torch.device, stream: int) -> torch.Tensor:
    """The zero-initialised workspace of the single-pass kernels for one
    device and stream (calls on one stream never overlap, so they may share
    it; the kernels leave it ready for the next call)."""
    key = (device.index, stream)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.zeros(_lib.SINGLE_PASS_WORKSPACE_BYTES, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def reset_workspaces() -> None:
    """Re-zeroes every cached workspace (after a reported device timeout)."""
    for ws in _workspaces.values():
        ws.zero_()


def scale_bytes(rows: int, cols: int, swizzled: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.load().nvfp4_scale_bytes(rows, cols, SWIZZLED if swizzled else 0, ctypes.byref(n)),
               "nvfp4_scale_bytes")
    return n.value


def compute_amax(x: torch.Tensor, amax_row: torch.Tensor, amax_col: torch.Tensor | None = None,
                 noop: torch.Tensor | None = None) -> None:
    """Zeroes amax_row (and amax_col) then writes max|x| into both."""
    _require_cuda(x, amax_row, amax_col, noop)
    M, N = (x.shape[0], x.numel() // x.shape[0]) if x.dim() > 0 and x.shape[0] > 0 else (0, 0)
    with _OnDevice(x.device):
        _lib.check(_lib.load().nvfp4_compute_amax(_ptr(x), _dtype_code(x), M, N, _ptr(amax_row), _ptr(amax_col),
                                                  _ptr(noop), _stream(x.device)), "nvfp4_compute_amax")


def compute_amax_rht(x: torch.Tensor, sign_mask: int, amax_row: torch.Tensor, amax_col: torch.Tensor,
                     noop: torch.Tensor | None = None) -> None:
    """max|x| into amax_row and max|RHT(x)| into amax_col (BF16 x, M x N)."""
    _require_cuda(x, amax_row, amax_col, noop)
    M, N = x.shape
    with _OnDevice(x.device):
        _lib.check(_lib.load().nvfp4_compute_amax_rht(_ptr(x), _dtype_code(x), M, N, sign_mask & 0xFFFF,
                                                      _ptr(amax_row), _ptr(amax_col), _ptr(noop),
                                                      _stream(x.device)), "nvfp4_compute_amax_rht")


def quantize(x: torch.Tensor, mode: str = "1d", rowwise: bool = True, colwise: bool = True,
             swizzled: bool = False, sign_mask: int = 0, out: NVFP4Tensor | None = None,
             skip_amax: bool = False, noop: torch.Tensor | None = None, path: str = "auto",
             workspace: torch.Tensor | None = None) -> NVFP4Tensor:
    """NVFP4-quantizes the 2-D tensor x (bfloat16 or float32) on its device.

    path: "auto" | "single_pass" | "two_pass" (1d / 2d only; see the module
    docstring).  workspace: for the single-pass path, a zeroed uint8 CUDA
    tensor of at least 4096 bytes owned by the caller (default: one cached
    per device and stream)."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (M x N)")
    M, N = x.shape
    row_scaled = mode == "row_scaled"
    if row_scaled:
        colwise = False
    if out is None:
        out = empty(M, N, rowwise, colwise, row_scaled=row_scaled, swizzled=swizzled, device=x.device)
    out.swizzled = swizzled
    _require_cuda(x, out.data_row, out.scale_row, out.amax_row, out.data_col, out.scale_col, out.amax_col, noop)
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLED if swizzled else 0) | \
        (SKIP_AMAX if skip_amax else 0)
    L = _lib.load()
    st = out.c_struct()
    if path not in ("auto", "single_pass", "two_pass"):
        raise ValueError(f"unknown path {path!r}")
    # rht: the single-pass kernel reads x from HBM once but is not faster than
    # the two kernels on GB300 (its cast phase is arithmetic-bound), so "auto"
    # keeps the two-pass path for it
    single = (mode in ("1d", "2d") or (mode == "rht" and path == "single_pass")) and not skip_amax and \
        path != "two_pass"
    if path == "single_pass" and not single:
        raise ValueError("the single-pass path covers 1d / 2d / rht quantize without skip_amax")
    with _OnDevice(x.device):
        s = _stream(x.device)
        if single:
            ws = workspace if workspace is not None else single_pass_workspace(x.device, s.value)
            _require_cuda(ws)
            if mode == "rht":
                rc = L.nvfp4_quantize_rht_single_pass(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags,
                                                      sign_mask & 0xFFFF, _ptr(noop), _ptr(ws), s)
            else:
                fn = L.nvfp4_quantize_1d_single_pass if mode == "1d" else L.nvfp4_quantize_2d_single_pass
                rc = fn(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, _ptr(noop), _ptr(ws), s)
        elif mode == "1d":
            rc = L.nvfp4_quantize_1d(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, _ptr(noop), s)
        elif mode == "2d":
            rc = L.nvfp4_quantize_2d(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, _ptr(noop), s)
        elif mode == "rht":
            rc = L.nvfp4_quantize_rht(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, sign_mask & 0xFFFF,
                                      _ptr(noop), s)
        elif mode == "row_scaled":
            rc = L.nvfp4_quantize_row_scaled(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, _ptr(noop), s)
        else:
            raise ValueError(f"unknown mode {mode!r}")
    _lib.check(rc, f"nvfp4 quantize ({mode})")
    return out


class QuantizePlan:
    """A quantize call bound once to its tensors, for loops that repeat it.

    ``quantize`` checks and marshals its arguments on every call (about
    10 µs of Python); a plan does that once -- the C function, the pointers,
    the flags, the output struct and, for the single-pass path, the
    workspace -- and each call then only passes them to the library with the
    stream.  The tensors must stay allocated, at the same addresses, for the
    plan's lifetime (the plan keeps references to them).  Arguments as
    ``quantize``; ``out`` defaults to buffers allocated here.

        plan = QuantizePlan(x, "2d", swizzled=True)
        plan()            # on x's device's current stream
        plan(stream=s)    # a torch.cuda.Stream or a raw cudaStream_t handle
    """

    def __init__(self, x: torch.Tensor, mode: str = "1d", rowwise: bool = True, colwise: bool = True,
                 swizzled: bool = False, sign_mask: int = 0, out: NVFP4Tensor | None = None,
                 skip_amax: bool = False, noop: torch.Tensor | None = None, path: str = "auto",
                 workspace: torch.Tensor | None = None):
        if x.dim() != 2:
            raise ValueError("x must be 2-D (M x N)")
        M, N = x.shape
        if mode == "row_scaled":
            colwise = False
        if out is None:
            out = empty(M, N, rowwise, colwise, row_scaled=mode == "row_scaled", swizzled=swizzled,
                        device=x.device)
        out.swizzled = swizzled
        _require_cuda(x, out.data_row, out.scale_row, out.amax_row, out.data_col, out.scale_col, out.amax_col,
                      noop)
        if path not in ("auto", "single_pass", "two_pass"):
            raise ValueError(f"unknown path {path!r}")
        flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLED if swizzled else 0) | \
            (SKIP_AMAX if skip_amax else 0)
        single = (mode in ("1d", "2d") or (mode == "rht" and path == "single_pass")) and not skip_amax and \
            path != "two_pass"
        if path == "single_pass" and not single:
            raise ValueError("the single-pass path covers 1d / 2d / rht quantize without skip_amax")
        L = _lib.load()
        self.x, self.out, self.noop, self.device = x, out, noop, x.device
        self._st = out.c_struct()
        head = (_ptr(x), _dtype_code(x), M, N, ctypes.byref(self._st), flags)
        if single:
            dev = x.device if x.device.index is not None else torch.device("cuda", torch.cuda.current_device())
            self.ws = workspace if workspace is not None else \
                single_pass_workspace(dev, torch.cuda.current_stream(dev).cuda_stream)
            _require_cuda(self.ws)
            if mode == "rht":
                self._fn, self._args = L.nvfp4_quantize_rht_single_pass, head + (sign_mask & 0xFFFF, _ptr(noop),
                                                                                   _ptr(self.ws))
            else:
                fn = L.nvfp4_quantize_1d_single_pass if mode == "1d" else L.nvfp4_quantize_2d_single_pass
                self._fn, self._args = fn, head + (_ptr(noop), _ptr(self.ws))
        elif mode in ("1d", "2d", "row_scaled"):
            fn = {"1d": L.nvfp4_quantize_1d, "2d": L.nvfp4_quantize_2d,
                  "row_scaled": L.nvfp4_quantize_row_scaled}[mode]
            self._fn, self._args = fn, head + (_ptr(noop),)
        elif mode == "rht":
            self._fn, self._args = L.nvfp4_quantize_rht, head + (sign_mask & 0xFFFF, _ptr(noop))
        else:
            raise ValueError(f"unknown mode {mode!r}")
        self.mode = mode
        self._dev_index = x.device.index if x.device.index is not None else torch.cuda.current_device()

    def __call__(self, stream=None) -> NVFP4Tensor:
        if stream is None:
            stream = torch.cuda.current_stream(self.device).cuda_stream
        elif isinstance(stream, torch.cuda.Stream):
            stream = stream.cuda_stream
        if torch.cuda.current_device() != self._dev_index:
            with _OnDevice(self.device):
                rc = self._fn(*self._args, ctypes.c_void_p(stream))
        else:
            rc = self._fn(*self._args, ctypes.c_void_p(stream))
        if rc != 0:
            _lib.check(rc, f"nvfp4 quantize plan ({self.mode})")
        return self.out


def quantize_sr(x: torch.Tensor, rbits: torch.Tensor, mode: str = "1d", rowwise: bool = True,
                colwise: bool = True, swizzled: bool = False, out: NVFP4Tensor | None = None,
                skip_amax: bool = False, noop: torch.Tensor | None = None) -> NVFP4Tensor:
    """NVFP4 quantize (mode "1d" or "2d") with stochastically rounded codes.

    rbits: a uint8 CUDA tensor of x's shape, the random numbers (the library
    draws none): element (y, j) of x rounds to the upper neighbouring E2M1
    magnitude iff rbits[y, j] < 256 f, f its position between the two, in
    both outputs.  Scales, amax and layouts as ``quantize``."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (M x N)")
    if mode not in ("1d", "2d"):
        raise ValueError("stochastic rounding: mode '1d' or '2d'")
    if rbits.dtype != torch.uint8 or tuple(rbits.shape) != tuple(x.shape):
        raise ValueError("rbits must be a uint8 tensor of x's shape")
    M, N = x.shape
    if out is None:
        out = empty(M, N, rowwise, colwise, swizzled=swizzled, device=x.device)
    out.swizzled = swizzled
    _require_cuda(x, rbits, out.data_row, out.scale_row, out.amax_row, out.data_col, out.scale_col, out.amax_col,
                  noop)
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLED if swizzled else 0) | \
        (SKIP_AMAX if skip_amax else 0)
    L = _lib.load()
    st = out.c_struct()
    fn = L.nvfp4_quantize_1d_sr if mode == "1d" else L.nvfp4_quantize_2d_sr
    with _OnDevice(x.device):
        rc = fn(_ptr(x), _dtype_code(x), M, N, ctypes.byref(st), flags, _ptr(rbits), _ptr(noop), _stream(x.device))
    _lib.check(rc, f"nvfp4 stochastic-rounding quantize ({mode})")
    return out


def quantize_grouped(x: torch.Tensor, splits, mode: str = "1d", rowwise: bool = True, colwise: bool = True,
                     swizzled: bool = False, out: list[NVFP4Tensor] | None = None, skip_amax: bool = False,
                     noop: torch.Tensor | None = None, path: str = "auto",
                     workspace: torch.Tensor | None = None) -> list[NVFP4Tensor]:
    """Grouped (multi-tensor) quantize: x (M x N, bfloat16 or float32) stacks
    len(splits) member tensors along its first dimension, member g being the
    splits[g] rows after the earlier members'.  Each member is quantized as a
    tensor of its own (its own amax, its own transpose) into its own
    NVFP4Tensor.  mode: "1d" or "2d".  out: one NVFP4Tensor per member
    (default: allocated).  path: "single_pass" (one persistent kernel, x read
    from HBM once; bfloat16, no skip_amax; the workspace as for ``quantize``),
    "three_pass" (zero the amaxes, max|x| per member, cast) or "auto" (single
    pass where it applies)."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D (M x N)")
    if mode not in ("1d", "2d"):
        raise ValueError("grouped quantize: mode '1d' or '2d'")
    splits = [int(m) for m in splits]
    if not 1 <= len(splits) <= _lib.MAX_GROUPS:
        raise ValueError(f"grouped quantize: 1 to {_lib.MAX_GROUPS} members")
    if sum(splits) != x.shape[0]:
        raise ValueError("grouped quantize: splits must sum to the rows of x")
    N = x.shape[1]
    if out is None:
        out = [empty(m, N, rowwise, colwise, swizzled=swizzled, device=x.device) for m in splits]
    if len(out) != len(splits):
        raise ValueError("grouped quantize: one output per member")
    for q in out:
        q.swizzled = swizzled
        _require_cuda(q.data_row, q.scale_row, q.amax_row, q.data_col, q.scale_col, q.amax_col)
    _require_cuda(x, noop)
    flags = (ROWWISE if rowwise else 0) | (COLWISE if colwise else 0) | (SWIZZLED if swizzled else 0) | \
        (SKIP_AMAX if skip_amax else 0)
    if path not in ("auto", "single_pass", "three_pass"):
        raise ValueError(f"unknown path {path!r}")
    single = x.dtype == torch.bfloat16 and not skip_amax and path != "three_pass"
    if path == "single_pass" and not single:
        raise ValueError("the single-pass grouped quantize takes bfloat16 x and no skip_amax")
    rows = (ctypes.c_int64 * len(splits))(*splits)
    outs = (_lib.Output * len(out))(*[q.c_struct() for q in out])
    L = _lib.load()
    with _OnDevice(x.device):
        s = _stream(x.device)
        if single:
            ws = workspace if workspace is not None else single_pass_workspace(x.device, s.value)
            _require_cuda(ws)
            fn = L.nvfp4_quantize_grouped_1d_single_pass if mode == "1d" else L.nvfp4_quantize_grouped_2d_single_pass
            rc = fn(_ptr(x), _dtype_code(x), N, len(splits), rows, outs, flags, _ptr(noop), _ptr(ws), s)
        else:
            fn = L.nvfp4_quantize_grouped_1d if mode == "1d" else L.nvfp4_quantize_grouped_2d
            rc = fn(_ptr(x), _dtype_code(x), N, len(splits), rows, outs, flags, _ptr(noop), s)
    _lib.check(rc, f"nvfp4 grouped quantize ({mode})")
    return out


def quantize_1d(x, **kw):
    return quantize(x, "1d", **kw)


def quantize_2d(x, **kw):
    return quantize(x, "2d", **kw)


def quantize_rht(x, sign_mask: int, **kw):
    return quantize(x, "rht", sign_mask=sign_mask, **kw)


def quantize_row_scaled(x, **kw):
    return quantize(x, "row_scaled", **kw)


def dequantize(data: torch.Tensor, scale: torch.Tensor, amax: torch.Tensor, swizzled: bool = False,
               row_scaled: bool = False, out_dtype: torch.dtype = torch.bfloat16,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """Dequantizes one direction: data [rows, cols/2] -> [rows, cols]."""
    rows, half = data.shape
    cols = 2 * half
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype, device=data.device)
    _require_cuda(data, scale, amax, out)
    od = BF16 if out.dtype == torch.bfloat16 else FP32 if out.dtype == torch.float32 else -1
    flags = (SWIZZLED if swizzled else 0) | (ROW_SCALED if row_scaled else 0)
    with _OnDevice(data.device):
        _lib.check(_lib.load().nvfp4_dequantize(_ptr(data), _ptr(scale), _ptr(amax), rows, cols, flags, _ptr(out), od,
                                                _stream(data.device)), "nvfp4_dequantize")
    return out


def swizzle_scales(compact: torch.Tensor, rows: int, scale_cols: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Compact [rows][scale_cols] scales -> the cuBLAS 128x4 layout (flat)."""
    if out is None:
        out = torch.empty(rows * scale_cols, dtype=torch.uint8, device=compact.device)
    _require_cuda(compact, out)
    with _OnDevice(compact.device):
        _lib.check(_lib.load().nvfp4_swizzle_scales(_ptr(compact), _ptr(out), rows, scale_cols,
                                                    _stream(compact.device)), "nvfp4_swizzle_scales")
    return out


def device_status(clear: bool = True) -> int:
    """Synchronizes the current device and returns its status word (0 = no
    device-side wait ran out)."""
    v = ctypes.c_uint32(0)
    rc = _lib.load().nvfp4_device_status(ctypes.byref(v), int(clear))
    if rc not in (0, 7):
        _lib.check(rc, "nvfp4_device_status")
    return v.value
