"""The C ABI without a GPU: the library builds and loads, exports every
function include/nvfp4.h declares, and rejects bad arguments with the
documented status before touching CUDA (validation is host-only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_FLAGS, ERR_CUDA = 0, 1, 2, 3, 4, 5, 6
ROW, COL, SWZ, SKIP, ROWSC = 1, 2, 4, 8, 16

# The calls below pass fake device addresses, so they must never reach a
# launch: the module does not run where a GPU is visible, and on a machine
# without one the fixture fails any call that got past validation (it then
# stops at the CUDA context, NVFP4_ERR_CUDA).
pytestmark = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="validation-only tests with fake device addresses: run on a machine without a GPU")

HOST_ONLY = ("nvfp4_status_string", "nvfp4_scale_bytes")


class _ValidationOnly:
    """The library, with every device entry point checked to fail validation."""

    def __init__(self, lib):
        self._lib = lib

    def __getattr__(self, name):
        fn = getattr(self._lib, name)
        if not name.startswith("nvfp4_") or name in HOST_ONLY:
            return fn

        def call(*args):
            rc = fn(*args)
            if rc == ERR_CUDA:
                pytest.fail(f"{name} accepted fake device addresses (it would launch on a GPU machine)")
            return rc
        return call


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_amax_gb300 import _lib, build
    build.build()
    return _ValidationOnly(_lib.load())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("nvfp4_compute_amax", "nvfp4_quantize_1d", "nvfp4_quantize_2d", "nvfp4_quantize_row_scaled",
                     "nvfp4_quantize_rht", "nvfp4_dequantize", "nvfp4_swizzle_scales"):
        assert required in names


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_compiles_for_c_and_cpp_hosts(tmp_path, lang, std):
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "nvfp4.h"\nint main(void) { nvfp4_output o; (void)o; '
                   'return (int)NVFP4_MAX_GROUPS - 64; }\n')
    subprocess.check_call([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                           "-I", os.path.join(ROOT, "include"), str(src)])


def test_library_exports_every_declared_function(lib):
    from nvfp4_block_scaled_amax_gb300 import _lib
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in nvfp4.h but not exported"
    assert set(names) <= set(_lib.EXPORTS) | set(names)
    assert sorted(_lib.EXPORTS) == names


def test_status_strings(lib):
    for code in range(8):
        s = lib.nvfp4_status_string(code).decode()
        assert s.startswith("NVFP4_")
    assert "unknown" in lib.nvfp4_status_string(99).decode()


def test_scale_bytes(lib):
    n = ctypes.c_size_t()
    assert lib.nvfp4_scale_bytes(256, 512, 0, ctypes.byref(n)) == OK and n.value == 256 * 32
    assert lib.nvfp4_scale_bytes(256, 512, SWZ, ctypes.byref(n)) == OK and n.value == 256 * 32
    assert lib.nvfp4_scale_bytes(200, 512, SWZ, ctypes.byref(n)) == ERR_ALIGN
    assert lib.nvfp4_scale_bytes(256, 24, 0, ctypes.byref(n)) == ERR_SHAPE
    assert lib.nvfp4_scale_bytes(256, 32, 0, None) == ERR_NULL


# Fake, 16-byte aligned device addresses: validation never dereferences them.
# Every call in this file must FAIL validation: one that passed would launch
# kernels on these addresses on a machine with a GPU (valid argument sets are
# exercised by the GPU tests, on real buffers).
X, A, B, C, D, E, F, NOOP = (0x100000 * (i + 1) for i in range(8))


def out(lib_mod, **kw):
    from nvfp4_block_scaled_amax_gb300._lib import Output
    base = dict(data_row=A, scale_row=B, amax_row=C, data_col=D, scale_col=E, amax_col=F)
    base.update(kw)
    return Output(**base)


def q1d(lib, x=X, dtype=0, M=256, N=256, o=None, flags=ROW | COL, noop=None):
    o = out(lib) if o is None else o
    return lib.nvfp4_quantize_1d(x, dtype, M, N, ctypes.byref(o), flags, noop, None)


def test_quantize_validation(lib):
    assert lib.nvfp4_quantize_1d(X, 0, 256, 256, None, ROW, None, None) == ERR_NULL
    assert q1d(lib, flags=0) == ERR_FLAGS                        # no direction
    assert q1d(lib, flags=ROW | 64) == ERR_FLAGS                 # unknown bit
    assert q1d(lib, flags=ROW | ROWSC) == ERR_FLAGS              # dequant-only flag
    assert q1d(lib, dtype=2) == ERR_DTYPE
    assert q1d(lib, M=-1) == ERR_SHAPE
    assert q1d(lib, N=24, flags=ROW) == ERR_SHAPE                # row blocks need N % 16
    assert q1d(lib, M=24, flags=COL) == ERR_SHAPE                # column blocks need M % 16
    # N % 16 whatever the directions: x is staged through a tensor map (row
    # pitch a multiple of 16 bytes) and the BF16 casts own 16 columns per lane
    assert q1d(lib, N=24, flags=COL) == ERR_SHAPE
    assert q1d(lib, dtype=1, N=20, flags=COL) == ERR_SHAPE
    assert q1d(lib, N=8, flags=COL | SKIP) == ERR_SHAPE
    assert lib.nvfp4_quantize_1d_single_pass(X, 0, 256, 24, ctypes.byref(out(lib)), COL, None, A, None) == ERR_SHAPE
    assert lib.nvfp4_quantize_2d_single_pass_noalloc(X, 0, 256, 40, ctypes.byref(out(lib)), COL, None,
                                                     None) == ERR_SHAPE
    assert q1d(lib, x=X + 8) == ERR_ALIGN
    assert q1d(lib, o=out(lib, data_col=D + 4)) == ERR_ALIGN
    assert q1d(lib, o=out(lib, scale_row=0)) == ERR_NULL
    assert q1d(lib, o=out(lib, amax_col=C)) == ERR_FLAGS          # aliased amax buffers
    assert q1d(lib, M=192, flags=ROW | COL | SWZ) == ERR_ALIGN    # swizzle needs 128-aligned
    assert q1d(lib, noop=NOOP + 4) == ERR_ALIGN
    assert q1d(lib, x=0) == ERR_NULL
    o = out(lib)
    assert lib.nvfp4_quantize_2d(X, 0, 256, 24, ctypes.byref(o), ROW, None, None) == ERR_SHAPE
    assert lib.nvfp4_quantize_2d(X, 0, 24, 256, ctypes.byref(o), ROW, None, None) == ERR_SHAPE
    assert lib.nvfp4_quantize_rht(X, 1, 256, 256, ctypes.byref(o), ROW | COL, 0, None, None) == ERR_DTYPE
    assert lib.nvfp4_quantize_row_scaled(X, 0, 256, 256, ctypes.byref(o), ROW | COL, None, None) == ERR_FLAGS
    assert lib.nvfp4_quantize_row_scaled(X, 0, 256, 256, ctypes.byref(o), COL, None, None) == ERR_FLAGS


def test_single_pass_validation(lib):
    o = out(lib)
    for fn in (lib.nvfp4_quantize_1d_single_pass, lib.nvfp4_quantize_2d_single_pass):
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | COL, None, None, None) == ERR_NULL        # workspace
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | COL, None, A + 4, None) == ERR_ALIGN
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | SKIP, None, A, None) == ERR_FLAGS        # no skip-amax
        assert fn(X, 0, 192, 256, ctypes.byref(o), ROW | COL | SWZ, None, A, None) == ERR_ALIGN
    assert lib.nvfp4_quantize_2d_single_pass(X, 0, 24, 256, ctypes.byref(o), ROW, None, A, None) == ERR_SHAPE
    rht = lib.nvfp4_quantize_rht_single_pass
    assert rht(X, 0, 256, 256, ctypes.byref(o), ROW | COL, 0, None, None, None) == ERR_NULL      # workspace
    assert rht(X, 0, 256, 256, ctypes.byref(o), ROW | COL, 0, None, A + 4, None) == ERR_ALIGN
    assert rht(X, 0, 256, 256, ctypes.byref(o), ROW | COL | SKIP, 0, None, A, None) == ERR_FLAGS
    assert rht(X, 1, 256, 256, ctypes.byref(o), ROW | COL, 0, None, A, None) == ERR_DTYPE       # BF16 only
    assert rht(X, 0, 24, 256, ctypes.byref(o), ROW | COL, 0, None, A, None) == ERR_SHAPE
    assert rht(X, 0, 192, 256, ctypes.byref(o), ROW | COL | SWZ, 0, None, A, None) == ERR_ALIGN


def test_amax_and_misc_validation(lib):
    assert lib.nvfp4_compute_amax(X, 0, 16, 16, None, None, None, None) == ERR_NULL
    assert lib.nvfp4_compute_amax(X, 0, 16, 16, C, C, None, None) == ERR_FLAGS
    assert lib.nvfp4_compute_amax(X, 3, 16, 16, C, None, None, None) == ERR_DTYPE
    assert lib.nvfp4_compute_amax(X + 2, 0, 16, 16, C, None, None, None) == ERR_ALIGN
    assert lib.nvfp4_compute_amax_rht(X, 0, 24, 16, 0, C, F, None, None) == ERR_SHAPE
    assert lib.nvfp4_compute_amax_rht(X, 1, 16, 16, 0, C, F, None, None) == ERR_DTYPE
    assert lib.nvfp4_dequantize(A, B, C, 128, 24, 0, D, 0, None) == ERR_SHAPE
    assert lib.nvfp4_dequantize(A, B, C, 120, 128, SWZ, D, 0, None) == ERR_ALIGN
    assert lib.nvfp4_dequantize(A, B, C, 128, 128, 2, D, 0, None) == ERR_FLAGS
    assert lib.nvfp4_dequantize(A, B, C, 128, 128, 0, D, 5, None) == ERR_DTYPE
    assert lib.nvfp4_dequantize(A, 0, C, 128, 128, 0, D, 0, None) == ERR_NULL
    assert lib.nvfp4_swizzle_scales(A, B, 100, 8, None) == ERR_ALIGN
    assert lib.nvfp4_swizzle_scales(A, B, 128, 6, None) == ERR_ALIGN
    assert lib.nvfp4_swizzle_scales(0, B, 128, 8, None) == ERR_NULL
    assert lib.nvfp4_device_status(None, 0) == ERR_NULL


def test_sr_validation(lib):
    o = out(lib)
    for fn in (lib.nvfp4_quantize_1d_sr, lib.nvfp4_quantize_2d_sr):
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | COL, None, None, None) == ERR_NULL     # random bytes
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | COL, A + 8, None, None) == ERR_ALIGN
        assert fn(X, 0, 256, 256, ctypes.byref(o), ROW | ROWSC, A, None, None) == ERR_FLAGS
        assert fn(X, 2, 256, 256, ctypes.byref(o), ROW, A, None, None) == ERR_DTYPE
        assert fn(X, 0, 256, 24, ctypes.byref(o), COL, A, None, None) == ERR_SHAPE            # N % 16 always
        assert fn(X, 0, 192, 256, ctypes.byref(o), ROW | SWZ, A, None, None) == ERR_ALIGN
        assert fn(X, 0, 256, 256, None, ROW, A, None, None) == ERR_NULL
    assert lib.nvfp4_quantize_2d_sr(X, 0, 24, 256, ctypes.byref(o), ROW, A, None, None) == ERR_SHAPE


def test_grouped_validation(lib):
    from nvfp4_block_scaled_amax_gb300._lib import Output

    def members(n, over=None):
        over = over or {}
        outs = (Output * n)()
        for g in range(n):
            base = 0x1000000 * (g + 1)
            d = dict(data_row=base, scale_row=base + 0x100000, amax_row=base + 0x200000,
                     data_col=base + 0x300000, scale_col=base + 0x400000, amax_col=base + 0x500000)
            d.update(over.get(g, {}))
            outs[g] = Output(**d)
        return outs

    def grouped(rows, o=None, fn=lib.nvfp4_quantize_grouped_1d, x=X, dtype=0, N=256, flags=ROW | COL, n=None,
                noop=None):
        r = (ctypes.c_int64 * len(rows))(*rows)
        o = members(len(rows)) if o is None else o
        return fn(x, dtype, N, len(rows) if n is None else n, r, o, flags, noop, None)

    r = (ctypes.c_int64 * 1)(128)
    assert lib.nvfp4_quantize_grouped_1d(X, 0, 256, 1, None, members(1), ROW, None, None) == ERR_NULL
    assert lib.nvfp4_quantize_grouped_1d(X, 0, 256, 1, r, None, ROW, None, None) == ERR_NULL
    assert grouped([128], n=0) == ERR_SHAPE                          # at least one member
    assert grouped([128] * 65) == ERR_SHAPE                          # at most 64
    assert grouped([128, -16]) == ERR_SHAPE
    assert grouped([128, 24]) == ERR_SHAPE                           # column blocks need rows % 16
    assert grouped([128, 24], flags=ROW, fn=lib.nvfp4_quantize_grouped_2d) == ERR_SHAPE
    assert grouped([128], N=24, flags=ROW) == ERR_SHAPE
    assert grouped([128], dtype=2) == ERR_DTYPE
    assert grouped([128], flags=0) == ERR_FLAGS
    assert grouped([128], flags=ROW | ROWSC) == ERR_FLAGS
    assert grouped([128, 64], flags=ROW | COL | SWZ) == ERR_ALIGN     # swizzle needs 128-row members
    assert grouped([128], x=X + 8) == ERR_ALIGN
    assert grouped([128], x=0) == ERR_NULL
    assert grouped([128, 128], o=members(2, {1: dict(scale_col=0)})) == ERR_NULL
    assert grouped([128, 128], o=members(2, {1: dict(data_row=0x7)})) == ERR_ALIGN
    shared = members(2, {1: dict(amax_row=0x1000000 + 0x200000)})  # member 1 reuses member 0's amax
    assert grouped([128, 128], o=shared) == ERR_FLAGS
    assert grouped([128], o=members(1, {0: dict(amax_col=0x1000000 + 0x200000)})) == ERR_FLAGS
    assert grouped([128], noop=NOOP + 4) == ERR_ALIGN

    # the single-launch form: the same checks, then BF16 only, no SKIP_AMAX,
    # and a 16-byte aligned workspace
    for fn in (lib.nvfp4_quantize_grouped_1d_single_pass, lib.nvfp4_quantize_grouped_2d_single_pass):
        def sp(rows, dtype=0, flags=ROW | COL, ws=A, o=None, x=X):
            r = (ctypes.c_int64 * len(rows))(*rows)
            o = members(len(rows)) if o is None else o
            return fn(x, dtype, 256, len(rows), r, o, flags, None, ws, None)
        assert sp([128, 24]) == ERR_SHAPE
        assert sp([128] * 65) == ERR_SHAPE
        assert sp([128], dtype=1) == ERR_DTYPE                        # FP32: the three-launch entry points
        assert sp([128], flags=ROW | COL | SKIP) == ERR_FLAGS           # a given amax: the three-launch form
        assert sp([128], ws=None) == ERR_NULL
        assert sp([128], ws=A + 4) == ERR_ALIGN
        assert sp([128, 64], flags=ROW | COL | SWZ) == ERR_ALIGN
        assert sp([128, 128], o=members(2, {1: dict(amax_row=0x1000000 + 0x200000)})) == ERR_FLAGS
        assert sp([128], x=X + 8) == ERR_ALIGN


def test_python_layer_rejects_cpu_tensors():
    import torch
    import nvfp4_block_scaled_amax_gb300 as nv
    x = torch.zeros(16, 16, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        nv.quantize(x, "1d", out=nv.NVFP4Tensor(16, 16, *(torch.zeros(1),) * 6))
    with pytest.raises(TypeError):
        nv._dtype_code(torch.zeros(16, 16, dtype=torch.float16))
