"""Row-slab sharding of one tensor's NVFP4 quantization over the ranks of a
torch.distributed group (one GPU per rank).

x (M x N) is split into row slabs; rank r quantizes rows [start_r, stop_r)
of x on its own GPU.  Per-tensor scaling couples the slabs only through the
amax: every rank reduces its slab, one MAX all-reduce of the vector
[error flag, amax_row, amax_col] combines them (the cross-rank amax
reduction that follows the local one, "Write both NVFP4 amax buffers",
Description), and every rank then casts its slab with the agreed amax
(SKIP_AMAX).  With RHT the vector carries the row amax and the amax after
the transform.  Row-scaled rows are independent tensors, so that mode needs
no exchange.  With stochastic rounding each rank passes the rows of the
random bytes that match its slab, so every element keeps its byte.

A rank's row-wise output is rows [start, stop) of the full row-wise output;
its column-wise output is columns [start/2, stop/2) of the packed codes of
x transposed (and the matching scale columns).  ``assemble`` joins the
ranks' parts into the buffers a single call on the whole tensor gives.

Failure handling stays on the host: a rank whose local step fails (a slab
the method does not define, a CUDA error) still joins the exchange with its
error flag set, so every rank raises ``ShardError`` instead of waiting for
it.  A rank that never joins makes the others' collective fail with the
process group's timeout.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch

from . import NVFP4Tensor, compute_amax, compute_amax_rht, empty, quantize, quantize_sr

__all__ = ["ShardError", "slab_bounds", "slab_alignment", "check_slab", "CudaBackend", "quantize_slab",
           "assemble", "all_reduce_max"]


class ShardError(RuntimeError):
    """A rank's slab could not be quantized; raised on every rank."""


def slab_alignment(mode: str, colwise: bool, swizzled: bool) -> int:
    """Row granularity of the slab boundaries: 128 for the 128x4 scale
    layout (whole scale tiles per rank), 16 where a column-wise block or a
    16x16 tile spans rows, else 1."""
    if swizzled:
        return 128
    if colwise or mode in ("2d", "rht"):
        return 16
    return 1


def slab_bounds(M: int, world: int, rank: int, align: int) -> tuple[int, int]:
    """Rows [start, stop) of rank `rank`: the M rows cut into units of
    `align` rows (the last may be short), dealt out as evenly as possible
    in rank order."""
    if world <= 0 or not 0 <= rank < world or align <= 0 or M < 0:
        raise ValueError("bad slab request")
    units = -(-M // align)
    per, extra = divmod(units, world)
    first = rank * per + min(rank, extra)
    count = per + (1 if rank < extra else 0)
    return min(M, first * align), min(M, (first + count) * align)


def check_slab(M_local: int, N: int, mode: str, rowwise: bool, colwise: bool, swizzled: bool) -> None:
    """Raises ValueError for a slab the method does not define."""
    if mode not in ("1d", "2d", "rht", "row_scaled"):
        raise ValueError(f"unknown mode {mode!r}")
    if mode == "row_scaled" and colwise:
        raise ValueError("row-scaled quantization is row-wise only")
    if not rowwise and not colwise:
        raise ValueError("nothing to produce")
    if rowwise and N % 16:
        raise ValueError(f"row-wise output needs N % 16 == 0 (N = {N})")
    if (colwise or mode in ("2d", "rht")) and M_local % 16:
        raise ValueError(f"slab of {M_local} rows: column blocks and 16x16 tiles need a multiple of 16")
    if swizzled and (M_local % 128 or N % 128):
        raise ValueError(f"swizzled scales need slabs of whole 128-row tiles and N % 128 == 0 "
                         f"({M_local} x {N})")


def all_reduce_max(vals: torch.Tensor, group=None) -> torch.Tensor:
    """MAX all-reduce of a small float32 vector over `group` (NCCL: on the
    device; other backends: through host memory)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return vals
    t = vals if dist.get_backend(group) == "nccl" else vals.cpu()
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return t.to(vals.device)


class CudaBackend:
    """The library's kernels on the slab's GPU."""

    def local_amax(self, x: torch.Tensor, mode: str, sign_mask: int) -> torch.Tensor:
        a = torch.zeros(8, dtype=torch.float32, device=x.device)  # two 16-byte aligned slots
        if mode == "rht":
            compute_amax_rht(x, sign_mask, a[0:1], a[4:5])
        else:
            compute_amax(x, a[0:1], a[4:5])
        return a[0::4]

    def cast(self, x: torch.Tensor, mode: str, amax: torch.Tensor, rowwise: bool, colwise: bool,
             swizzled: bool, sign_mask: int, rbits: torch.Tensor | None = None) -> NVFP4Tensor:
        M, N = x.shape
        out = empty(M, N, rowwise, colwise, swizzled=swizzled, device=x.device)
        if out.amax_row is not None:
            out.amax_row.copy_(amax[0:1])
        if out.amax_col is not None:
            out.amax_col.copy_(amax[1:2])
        if rbits is not None:
            return quantize_sr(x, rbits, mode, rowwise=rowwise, colwise=colwise, swizzled=swizzled, out=out,
                               skip_amax=True)
        return quantize(x, mode, rowwise=rowwise, colwise=colwise, swizzled=swizzled, sign_mask=sign_mask,
                        out=out, skip_amax=True)

    def quantize_rows(self, x: torch.Tensor, swizzled: bool) -> NVFP4Tensor:
        return quantize(x, "row_scaled", rowwise=True, colwise=False, swizzled=swizzled)


def quantize_slab(x_local: torch.Tensor, mode: str = "1d", *, rowwise: bool = True, colwise: bool = True,
                  swizzled: bool = False, sign_mask: int = 0, group=None, backend=None,
                  exchange: Callable[[torch.Tensor], torch.Tensor] | None = None,
                  rbits_local: torch.Tensor | None = None) -> NVFP4Tensor:
    """Quantizes this rank's row slab of a tensor split over the ranks.

    Every rank of the group calls this with its slab (the same N, mode and
    flags).  `rbits_local`: stochastic rounding of the codes (modes 1d and
    2d), the rows of the random bytes that match the slab.  `exchange` replaces the MAX all-reduce over `group` (it gets
    and returns the float32 vector [error, amax_row, amax_col]); `backend`
    replaces the library's kernels.  Raises ShardError on every rank when
    any rank's slab fails its local step."""
    backend = backend if backend is not None else CudaBackend()
    exchange = exchange if exchange is not None else (lambda v: all_reduce_max(v, group))
    if x_local.dim() != 2:
        raise ValueError("x_local must be 2-D")
    M_local, N = x_local.shape
    if rbits_local is not None and (mode not in ("1d", "2d") or tuple(rbits_local.shape) != (M_local, N)):
        raise ValueError("rbits_local: modes 1d / 2d, one byte per element of the slab")
    if mode == "row_scaled":
        check_slab(M_local, N, mode, rowwise, False, swizzled)
        return backend.quantize_rows(x_local, swizzled)

    err, amax, why = 0.0, None, ""
    try:
        check_slab(M_local, N, mode, rowwise, colwise, swizzled)
        amax = backend.local_amax(x_local, mode, sign_mask).to(torch.float32).reshape(2)
    except Exception as e:  # joined below so that no rank waits for this one
        err, why = 1.0, f"{type(e).__name__}: {e}"
    vals = torch.zeros(3, dtype=torch.float32, device=x_local.device)
    vals[0] = err
    if amax is not None:
        vals[1:3] = amax.to(vals.device)
    vals = exchange(vals)
    if float(vals[0]) != 0.0:
        raise ShardError(f"this rank's slab failed ({why})" if why else "another rank's slab failed")
    if rbits_local is not None:
        return backend.cast(x_local, mode, vals[1:3], rowwise, colwise, swizzled, sign_mask, rbits=rbits_local)
    return backend.cast(x_local, mode, vals[1:3], rowwise, colwise, swizzled, sign_mask)


def assemble(parts: Sequence[NVFP4Tensor]) -> NVFP4Tensor:
    """The buffers of the whole tensor from the ranks' parts (rank order).

    Row-wise data and scales are row ranges, so they concatenate; column-
    wise codes and compact scales are column ranges of the transposed
    output; in the 128x4 layout a part's column scales are whole 4-column
    groups of every 128-row band, so they interleave band by band."""
    if not parts:
        raise ValueError("no parts")
    N, swz, rs = parts[0].N, parts[0].swizzled, parts[0].row_scaled
    if any(p.N != N or p.swizzled != swz or p.row_scaled != rs for p in parts):
        raise ValueError("parts of different tensors")
    M = sum(p.M for p in parts)
    q = NVFP4Tensor(M, N, swizzled=swz, row_scaled=rs)
    if parts[0].data_row is not None:
        q.data_row = torch.cat([p.data_row for p in parts], 0)
        q.scale_row = torch.cat([p.scale_row for p in parts], 0)
        q.amax_row = torch.cat([p.amax_row for p in parts], 0) if rs else parts[0].amax_row.clone()
    if parts[0].data_col is not None:
        q.data_col = torch.cat([p.data_col for p in parts], 1)
        if swz:
            q.scale_col = torch.cat([p.scale_col.view(N // 128, -1, 512) for p in parts], 1).reshape(-1)
        else:
            q.scale_col = torch.cat([p.scale_col.view(N, -1) for p in parts], 1).reshape(-1)
        q.amax_col = parts[0].amax_col.clone()
    return q
