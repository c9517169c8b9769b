"""The entry point that allocates nothing (nvfp4_quantize_2d_single_pass_noalloc).

Some callers cannot allocate device memory: a plain C host that embeds the
library with no device memory manager, code that must not take an
allocator's lock or risk a synchronizing cudaMalloc / cudaFree, or a process
that sized all of its device memory up front.  For them the library keeps
the single-pass kernel's scratch in a static array of its own.  This test
calls that entry point through the C ABI twice in a row (the array keeps
the previous call's contents) and checks each result against the regular
single-pass entry point, which uses a caller-allocated workspace, and
against the oracle.  It lives
in its own file, collected last, so a run that stops at the first failure
has already run every other test.
"""
import ctypes

import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import _lib, inputs
from nvfp4_testutil import assert_quantize_equal, bits

pytestmark = pytest.mark.gpu

ROW, COL, SWZ = 1, 2, 4


def _outputs(M, N):
    return nv.empty(M, N, device="cuda")


def _noalloc(x, q, flags):
    st = q.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _lib.load().nvfp4_quantize_2d_single_pass_noalloc(ctypes.c_void_p(x.data_ptr()), 0, x.shape[0], x.shape[1],
                                                           ctypes.byref(st), flags, None, stream)
    assert rc == 0, _lib.load().nvfp4_status_string(rc).decode()


def _same(a, b):
    for name in ("data_row", "scale_row", "amax_row", "data_col", "scale_col", "amax_col"):
        ta, tb = getattr(a, name), getattr(b, name)
        assert torch.equal(ta, tb), name   # the 2D codec is exact: no tolerance


def test_noalloc_matches_single_pass_on_consecutive_calls(oracle_mod):
    torch.cuda.set_device(0)
    M, N = 2048, 1536
    x1 = inputs.outliers(M, N, seed=41, frac=0.01)
    x2 = (inputs.randn(M, N, seed=42) * 0.25).to(torch.bfloat16)   # a smaller maximum
    for step, xh in enumerate((x1, x2)):     # two calls in a row on the shared array
        x = xh.cuda()
        got = _outputs(M, N)
        _noalloc(x, got, ROW | COL | SWZ)
        ref = nv.quantize(x, "2d", swizzled=True, path="single_pass")
        torch.cuda.synchronize()
        _same(got, ref)
        assert_quantize_equal(oracle_mod, got, oracle_mod.quantize("2d", bits(xh)), True, what=f"no-alloc call {step}")


def test_noalloc_rejects_bad_arguments_without_launching():
    q = _outputs(256, 256)
    st = q.c_struct()
    L = _lib.load()
    x = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    # swizzled scales on a shape that is not 128-aligned: refused on the host
    rc = L.nvfp4_quantize_2d_single_pass_noalloc(ctypes.c_void_p(x.data_ptr()), 0, 192, 256, ctypes.byref(st),
                                                 ROW | COL | SWZ, None, None)
    assert rc == 3
