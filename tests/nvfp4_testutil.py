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


def compare_rht_codes(got_data: np.ndarray, ref_data: np.ndarray, got_scale: np.ndarray, ref_scale: np.ndarray):
    """Column-wise RHT outputs: codes may differ from the oracle by one E2M1
    step (the kernel sums the Hadamard products in butterfly order, the
    oracle in ascending order); returns (n_code_diffs, n_scale_diffs) after
    checking every difference is a single step of the same sign."""
    g, r = unpack(got_data), unpack(ref_data)
    diff = g != r
    if diff.any():
        gi, ri = g[diff], r[diff]
        same_sign = ((gi & 8) == (ri & 8)) | ((gi & 7) == 0) | ((ri & 7) == 0)
        one_step = np.abs((gi & 7).astype(int) - (ri & 7).astype(int)) == 1
        assert np.all(same_sign & one_step), "RHT code differs by more than one E2M1 step"
    sdiff = got_scale != ref_scale
    if sdiff.any():
        assert np.all(np.abs(got_scale[sdiff].astype(int) - ref_scale[sdiff].astype(int)) == 1), \
            "RHT scale differs by more than one E4M3 step"
    return int(diff.sum()), int(sdiff.sum())
