"""Shared helpers of the test-suite: building the GPU self-test library,
moving tensors to numpy, and comparing library outputs with the oracle."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SELFTEST_SRC = os.path.join(HERE, "gpu_selftest.cu")
SELFTEST_LIB = os.path.join(HERE, "_build", "libselftest.so")

E2M1_MAG = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def build_selftest() -> ctypes.CDLL:
    os.makedirs(os.path.dirname(SELFTEST_LIB), exist_ok=True)
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_amax_gb300", "csrc")
    deps = [SELFTEST_SRC, os.path.join(csrc, "common.cuh")]
    if not os.path.exists(SELFTEST_LIB) or any(os.path.getmtime(d) > os.path.getmtime(SELFTEST_LIB) for d in deps):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "--fmad=false", "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(ROOT, "include"),
                               "-I", csrc, SELFTEST_SRC, "-o", SELFTEST_LIB])
    L = ctypes.CDLL(SELFTEST_LIB)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.selftest_e2m1.argtypes = [vp, vp, i64]
    L.selftest_e4m3.argtypes = [vp, vp, i64]
    L.selftest_e2m1_sr.argtypes = [vp, vp, vp, i64]
    L.selftest_bf16.argtypes = [vp, vp, i64]
    L.selftest_div6.argtypes = [ctypes.c_uint32, ctypes.c_uint32, vp, vp]
    L.selftest_wait_timeout.argtypes = [vp, ctypes.c_longlong, vp]
    return L


def bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor -> uint16 numpy bit patterns (float32 -> float32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def np_(t: torch.Tensor | None) -> np.ndarray | None:
    return None if t is None else t.detach().cpu().numpy()


def unpack(data: np.ndarray) -> np.ndarray:
    """Packed codes [R, C/2] -> codes [R, C]."""
    q = np.empty((data.shape[0], data.shape[1] * 2), np.uint8)
    q[:, 0::2] = data & 0xF
    q[:, 1::2] = data >> 4
    return q


def code_value(q: np.ndarray) -> np.ndarray:
    return np.where(q & 8, -1.0, 1.0) * E2M1_MAG[q & 7]


def expected_scales(oracle, compact: np.ndarray, swizzled: bool) -> np.ndarray:
    return oracle.swizzle(compact) if swizzled else compact.reshape(-1)


def scales_compact(oracle, flat: np.ndarray, R: int, C: int, swizzled: bool) -> np.ndarray:
    """A scale buffer as a compact [R][C] array.  Swizzled buffers are read
    back through the oracle's own permutation: swizzling the four bytes of
    every element's compact index gives, at each stored position, the index
    of the scale stored there."""
    flat = np.asarray(flat).reshape(-1)
    if not swizzled:
        return flat.reshape(R, C)
    idx = np.arange(R * C, dtype=np.uint32).reshape(R, C)
    src = np.zeros(R * C, dtype=np.uint32)
    for k in range(4):
        plane = ((idx >> (8 * k)) & 0xFF).astype(np.uint8)
        src |= oracle.swizzle(plane).astype(np.uint32) << (8 * k)
    out = np.empty(R * C, dtype=np.uint8)
    out[src] = flat
    return out.reshape(R, C)


def assert_quantize_equal(oracle, q, ref: dict, swizzled: bool, rowwise=True, colwise=True, what=""):
    """Bit-exact comparison of a library NVFP4Tensor with oracle output."""
    if rowwise:
        np.testing.assert_array_equal(np_(q.amax_row), ref["amax_row"], err_msg=f"{what} amax_row")
        np.testing.assert_array_equal(np_(q.data_row), ref["row_data"], err_msg=f"{what} row data")
        np.testing.assert_array_equal(np_(q.scale_row), expected_scales(oracle, ref["row_scale"], swizzled),
                                      err_msg=f"{what} row scales")
    if colwise:
        np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"], err_msg=f"{what} amax_col")
        np.testing.assert_array_equal(np_(q.data_col), ref["col_data"], err_msg=f"{what} col data")
        np.testing.assert_array_equal(np_(q.scale_col), expected_scales(oracle, ref["col_scale"], swizzled),
                                      err_msg=f"{what} col scales")


def _bf16_f64(bits16: np.ndarray) -> np.ndarray:
    return (bits16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_toward(t16: np.ndarray, target: np.ndarray) -> np.ndarray:
    """The BF16 neighbour of each BF16 value t16 (float32 array) in the
    direction of target (t16 itself where target equals it)."""
    b = (t16.view(np.uint32) >> 16).astype(np.int64)
    neg = (b & 0x8000) != 0
    mag = b & 0x7FFF
    up = target > t16
    # away from zero: magnitude + 1; toward zero: magnitude - 1 (through 0 to
    # the smallest subnormal of the other sign)
    away = np.where(neg, ~up, up)
    new_mag = np.where(away, mag + 1, mag - 1)
    cross = (~away) & (mag == 0)
    new_b = np.where(cross, np.where(neg, 0x0001, 0x8001), (b & 0x8000) | np.maximum(new_mag, 0))
    new_b = np.where(target == t16, b, new_b)
    return (new_b.astype(np.uint32) << 16).view(np.float32)


def rht_tie_candidates(oracle, xb: np.ndarray, mask: int, cols: np.ndarray):
    """For the columns ``cols`` of x: the oracle's transformed values t (BF16,
    as float32, [len(cols), M]), each value's BF16 neighbour t' toward the
    exact transform S, and the tie candidates: where S lies within
    B = 32 u sum|terms| (u = 2^-24) of the midpoint of t and t', so that an
    FP32 sum taken in another order may round to t' instead of t."""
    M = xb.shape[0]
    H = oracle.hadamard16().astype(np.float64)
    sign = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    t16 = oracle.rht_columns(xb, mask, True, cols)                     # [k, M]
    X = _bf16_f64(xb[:, cols])                                         # [M, k]
    u = X.reshape(M // 16, 16, len(cols)) * sign[None, :, None]
    S = (np.einsum("oi,bin->bon", H, u) / 4.0).reshape(M, len(cols)).T  # exact transform
    B = 2.0 ** -19 * np.repeat(np.abs(u).sum(axis=1) / 4.0, 16, axis=0).T
    alt = _bf16_toward(t16, S)
    mid = (t16.astype(np.float64) + alt.astype(np.float64)) / 2.0
    cand = (alt != t16) & (np.abs(S - mid) <= B)
    return t16, alt, cand


def check_rht_columns(oracle, xb: np.ndarray, mask: int, got_data: np.ndarray, got_scale: np.ndarray,
                      ref: dict, cols: np.ndarray | None = None, chunk: int = 512,
                      cache: dict | None = None) -> dict:
    """Column-wise output of the Hadamard quantize against the oracle, under
    the stated tolerance: a code may differ from the oracle's only at a
    rounding tie of the transform, and a scale only where such a tie moves
    its block's maximum.

    The oracle sums each transformed value in FP32 in ascending order, the
    kernels in their own order (butterflies, tensor cores); both round the
    FP32 sum to BF16.  The products are exact, so the two sums lie within
    the error bound of a 16-term FP32 summation of the exact value S, taken
    here as B = 32 u sum|terms| (u = 2^-24; twice the textbook (n - 1) u
    sum|terms|, for accumulators that align before they round).  So the
    kernel's BF16 value is the oracle's t, or -- only where S lies within B
    of the midpoint between t and its BF16 neighbour t' toward S (a tie
    candidate) -- t'.  Checked exactly: every kernel code is E2M1(t r) or,
    at a tie candidate, E2M1(t' r), with r = g / float(s) from the kernel's
    own block scale s; every kernel scale lies between the block scales of
    the smallest and the largest block maximum those choices allow; codes
    equal up to the sign of a zero count as equal.  got_data [nc, M/2] and
    got_scale [nc, M/16] (compact) are the kernel's rows for the columns
    ``cols`` of x (all when None); ``ref`` the oracle's quantize output for
    the same columns.  Returns the counts (differing codes and scales, tie
    candidates) and the number of codes compared.  ``cache``: a dict kept by
    the caller between checks of the same x and mask (the transform and its
    tie candidates are then computed once)."""
    M, N = xb.shape
    ids = np.arange(N, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64)
    nc = ids.size
    g = oracle.global_encode_scale(float(ref["amax_col"][0]))
    rtab = np.array([oracle.encode_factor(s, g) for s in range(128)], dtype=np.float32)
    got_codes = unpack(got_data)
    ref_codes = unpack(ref["col_data"])
    got_scale = got_scale.reshape(nc, M // 16)
    ref_scale = ref["col_scale"].reshape(nc, M // 16)
    assert int(got_scale.max(initial=0)) < 128, "scale code outside E4M3's non-negative finite range"
    n_codes = n_scales = n_cand = 0
    for c0 in range(0, nc, chunk):
        sl = slice(c0, min(nc, c0 + chunk))
        cid = ids[sl]
        key = (c0, cid.size, mask)
        if cache is not None and key in cache:
            t16, alt, cand = cache[key]
        else:
            t16, alt, cand = rht_tie_candidates(oracle, xb, mask, cid)
            if cache is not None:
                cache[key] = (t16, alt, cand)
        n_cand += int(cand.sum())
        sg = got_scale[sl]
        r = np.repeat(rtab[sg], 16, axis=1)
        c_t = oracle.encode_array(t16 * r, "e2m1")
        c_a = oracle.encode_array(alt * r, "e2m1")
        gc, rc = got_codes[sl], ref_codes[sl]
        both_zero = ((gc & 7) == 0) & ((c_t & 7) == 0)
        explained = (gc == c_t) | (cand & (gc == c_a)) | both_zero
        bad = np.argwhere(~explained)
        assert bad.size == 0, (f"RHT column code not explained by a rounding tie at (column {cid[bad[0][0]]}, "
                               f"row {bad[0][1]}): kernel {gc[tuple(bad[0])]:#x}, oracle {rc[tuple(bad[0])]:#x}")
        same = sg == ref_scale[sl]
        rep = np.repeat(same, 16, axis=1)
        # the harness agrees with the oracle where the scales agree
        assert np.all((c_t == rc) | ~rep), "check_rht_columns disagrees with the oracle's own codes"
        n_codes += int(((gc != rc) & ~(((gc & 7) == 0) & ((rc & 7) == 0))).sum())
        for k, blk in np.argwhere(~same):
            lo_hi = slice(16 * blk, 16 * blk + 16)
            a, b = np.abs(t16[k, lo_hi]), np.abs(np.where(cand[k, lo_hi], alt[k, lo_hi], t16[k, lo_hi]))
            b_lo, b_hi = float(np.minimum(a, b).max()), float(np.maximum(a, b).max())
            allowed = {oracle.block_scale(b_lo, g), oracle.block_scale(b_hi, g)}
            assert int(sg[k, blk]) in allowed, (f"RHT column scale at (column {cid[k]}, block {blk}) is "
                                               f"{int(sg[k, blk]):#x}, not one of {sorted(allowed)}")
            n_scales += 1
    counts = {"codes_differing": n_codes, "scales_differing": n_scales, "tie_candidates": n_cand,
              "codes_compared": nc * M}
    print(f"RHT column-wise parity: {counts}")
    return counts


def oracle_quantize_slabs(oracle, mode: str, xb: np.ndarray, rowwise: bool = True, colwise: bool = True,
                          sign_mask: int = 0, workers: int | None = None) -> dict:
    """The oracle's quantization of the whole of x, as one ``oracle.quantize``
    call would return it, computed as slabs of output rows on a thread pool
    (the oracle is single-threaded C; ctypes releases the GIL during each
    call).  Each slab is an oracle call on the whole x that selects some rows
    of the row-wise output or some columns of x, with the tensor's amax pair
    given (``oracle.amax`` / ``oracle.rht_amax`` of x; row-scaled rows use
    their own).  Nothing is computed outside the oracle: this only splits the
    work and concatenates the slabs."""
    import concurrent.futures as cf

    M, N = xb.shape
    if mode == "row_scaled":
        amax = None
    elif mode == "rht":
        amax = (oracle.amax(xb), oracle.rht_amax(xb, sign_mask))
    else:
        a = oracle.amax(xb)
        amax = (a, a)
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    jobs = []
    if rowwise:
        for ids in np.array_split(np.arange(M, dtype=np.int64), max(1, min(M, 4 * workers))):
            if ids.size:
                jobs.append(("row", ids))
    if colwise:
        for ids in np.array_split(np.arange(N, dtype=np.int64), max(1, min(N, 4 * workers))):
            if ids.size:
                jobs.append(("col", ids))

    def run(job):
        kind, ids = job
        return oracle.quantize(mode, xb, rowwise=kind == "row", colwise=kind == "col", sign_mask=sign_mask,
                               amax=amax, rows=ids if kind == "row" else None, cols=ids if kind == "col" else None)

    with cf.ThreadPoolExecutor(workers) as ex:
        parts = list(ex.map(run, jobs))
    rows = [p for (k, _), p in zip(jobs, parts) if k == "row"]
    cols = [p for (k, _), p in zip(jobs, parts) if k == "col"]
    out = {"row_data": np.zeros((0, N // 2), np.uint8), "row_scale": np.zeros((0, N // 16), np.uint8),
           "col_data": np.zeros((0, M // 2), np.uint8), "col_scale": np.zeros((0, M // 16), np.uint8)}
    if rows:
        out["row_data"] = np.concatenate([p["row_data"] for p in rows])
        out["row_scale"] = np.concatenate([p["row_scale"] for p in rows])
        out["amax_row"] = np.concatenate([p["amax_row"] for p in rows]) if mode == "row_scaled" else \
            rows[0]["amax_row"]
    if cols:
        out["col_data"] = np.concatenate([p["col_data"] for p in cols])
        out["col_scale"] = np.concatenate([p["col_scale"] for p in cols])
        out["amax_col"] = cols[0]["amax_col"]
    if amax is not None:
        out.setdefault("amax_row", np.array([amax[0]], np.float32))
        out.setdefault("amax_col", np.array([amax[1]], np.float32))
    return out
