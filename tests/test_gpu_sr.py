"""Quantize with stochastically rounded codes against the oracle, bit for
bit: random bytes passed in (one per element of x, shared by both outputs),
1D / 2D, BF16 / FP32, row / column / both, compact and swizzled scales,
ragged tiles and ragged rows, skip-amax and noop, the scales equal to the
round-to-nearest path, and the full-size workload on sampled rows and
columns."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import assert_quantize_equal, bits, np_

pytestmark = pytest.mark.gpu

SHAPES = [(16, 16), (128, 128), (48, 80), (208, 336), (256, 384), (1088, 1024), (16, 4096), (4096, 16)]
FLAGS = [(True, True), (True, False), (False, True)]


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_sr_matches_oracle(oracle_mod, M, N, dtype, mode):
    x = inputs.outliers(M, N, seed=M * 3 + N, frac=0.01, dtype=dtype)
    rb = inputs.random_bytes(M, N, seed=M + 5 * N)
    xd, rbd = x.cuda(), rb.cuda()
    swz_ok = M % 128 == 0 and N % 128 == 0
    for rowwise, colwise in FLAGS:
        ref = oracle_mod.quantize(mode, bits(x), rowwise=rowwise, colwise=colwise, rbits=rb.numpy())
        for swizzled in ([False, True] if swz_ok else [False]):
            q = nv.quantize_sr(xd, rbd, mode, rowwise=rowwise, colwise=colwise, swizzled=swizzled)
            torch.cuda.synchronize()
            assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise, colwise,
                                  what=f"sr {mode} {M}x{N} {dtype} r{rowwise}c{colwise}s{swizzled}")
    assert nv.device_status() == 0


def test_sr_row_only_ragged_rows(oracle_mod):
    for M in (1, 40, 129):
        x = inputs.randn(M, 96, seed=M)
        rb = inputs.random_bytes(M, 96, seed=7 * M)
        ref = oracle_mod.quantize("1d", bits(x), colwise=False, rbits=rb.numpy())
        q = nv.quantize_sr(x.cuda(), rb.cuda(), "1d", colwise=False)
        torch.cuda.synchronize()
        assert_quantize_equal(oracle_mod, q, ref, False, colwise=False, what=f"sr row-only M={M}")


def test_sr_extreme_bytes_and_scales(oracle_mod):
    """Bytes 0 (every inexact product rounds away from zero) and 255, and
    the scales and amax equal to the round-to-nearest quantize."""
    M, N = 256, 384
    x = inputs.outliers(M, N, seed=17, frac=0.01)
    xd = x.cuda()
    plain = nv.quantize(xd, "1d", path="two_pass")
    for byte in (0, 255):
        rb = torch.full((M, N), byte, dtype=torch.uint8)
        q = nv.quantize_sr(xd, rb.cuda(), "1d")
        torch.cuda.synchronize()
        ref = oracle_mod.quantize("1d", bits(x), rbits=rb.numpy())
        assert_quantize_equal(oracle_mod, q, ref, False, what=f"sr byte {byte}")
        for a, b in ((q.scale_row, plain.scale_row), (q.scale_col, plain.scale_col), (q.amax_row, plain.amax_row),
                     (q.amax_col, plain.amax_col)):
            assert torch.equal(a, b)


def test_sr_skip_amax_and_noop(oracle_mod):
    M, N = 256, 256
    x = inputs.randn(M, N, seed=19)
    rb = inputs.random_bytes(M, N, seed=20)
    xd, rbd = x.cuda(), rb.cuda()
    a = oracle_mod.amax(bits(x))
    q = nv.empty(M, N, device="cuda")
    q.amax_row.fill_(2 * a)
    q.amax_col.fill_(3 * a)
    nv.quantize_sr(xd, rbd, "2d", out=q, skip_amax=True)
    torch.cuda.synchronize()
    ref = oracle_mod.quantize("2d", bits(x), amax=(2 * a, 3 * a), rbits=rb.numpy())
    assert_quantize_equal(oracle_mod, q, ref, False, what="sr skip-amax")
    for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
        t.fill_(0xAB)
    q.amax_row.fill_(-3.0)
    nv.quantize_sr(xd, rbd, "1d", out=q, noop=torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
        assert bool((t == 0xAB).all())
    assert q.amax_row.item() == -3.0


@pytest.mark.slow
def test_sr_full_size_sampled(oracle_mod):
    spec = inputs.SR
    M, N = spec["M"], spec["N"]
    x = inputs.make(spec)
    rb = inputs.random_bytes(M, N, seed=spec["rbits_seed"])
    q = nv.quantize_sr(x.cuda(), rb.cuda(), spec["mode"], swizzled=spec["swizzled"])
    torch.cuda.synchronize()
    xb = bits(x)
    assert np_(q.amax_row)[0] == oracle_mod.amax(xb) and np_(q.amax_col)[0] == oracle_mod.amax(xb)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([rng.choice(M, 24, replace=False), [0, M - 1]])).astype(np.int64)
    cols = np.unique(np.concatenate([rng.choice(N, 24, replace=False), [0, N - 1]])).astype(np.int64)
    ref = oracle_mod.quantize(spec["mode"], xb, rows=rows, cols=cols, rbits=rb.numpy())
    np.testing.assert_array_equal(np_(q.data_row)[rows], ref["row_data"])
    np.testing.assert_array_equal(np_(q.data_col)[cols], ref["col_data"])
    off_r = np.array([[oracle_mod.swizzle_offset(int(i), c, N // 16) for c in range(N // 16)] for i in rows])
    off_c = np.array([[oracle_mod.swizzle_offset(int(j), c, M // 16) for c in range(M // 16)] for j in cols])
    np.testing.assert_array_equal(np_(q.scale_row)[off_r], ref["row_scale"])
    np.testing.assert_array_equal(np_(q.scale_col)[off_c], ref["col_scale"])
    assert nv.device_status() == 0
