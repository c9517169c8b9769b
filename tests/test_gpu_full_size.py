"""Parity at the full workload sizes, in the launch configuration the
benchmark times: amax exactly, then sampled rows of the row-wise output and
sampled columns of x (rows of the column-wise output) against the oracle,
plus size-independent properties (swizzled = permuted compact, dequantize of
the sampled rows, the dual-amax reuse sequence)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import bits, compare_rht_codes, np_

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(n, k, seed, must=()):
    rng = np.random.default_rng(seed)
    s = set(int(v) for v in rng.choice(n, size=min(k, n), replace=False))
    s.update(int(m) for m in must if 0 <= m < n)
    return np.array(sorted(s), dtype=np.int64)


def _scale_rows(flat, rows, C, swizzled, oracle):
    """Scale bytes of the given rows, read from a compact or swizzled buffer."""
    if not swizzled:
        return flat.reshape(-1, C)[rows]
    off = np.array([[oracle.swizzle_offset(int(r), c, C) for c in range(C)] for r in rows], dtype=np.int64)
    return flat[off]


def _check_sampled(oracle, q, x_bits, mode, rows, cols, swizzled, sign_mask=0, exact_cols=True):
    M, N = x_bits.shape
    ref = oracle.quantize(mode, x_bits, rowwise=q.data_row is not None, colwise=q.data_col is not None,
                          sign_mask=sign_mask, rows=rows, cols=cols)
    if q.data_row is not None:
        np.testing.assert_array_equal(np_(q.amax_row)[:1] if mode != "row_scaled" else np_(q.amax_row)[rows],
                                      ref["amax_row"])
        np.testing.assert_array_equal(np_(q.data_row)[rows], ref["row_data"])
        np.testing.assert_array_equal(_scale_rows(np_(q.scale_row), rows, N // 16, swizzled, oracle),
                                      ref["row_scale"])
    if q.data_col is not None:
        np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"])
        got_d = np_(q.data_col)[cols]
        got_s = _scale_rows(np_(q.scale_col), cols, M // 16, swizzled, oracle)
        if exact_cols:
            np.testing.assert_array_equal(got_d, ref["col_data"])
            np.testing.assert_array_equal(got_s, ref["col_scale"])
        else:
            nd, ns = compare_rht_codes(got_d, ref["col_data"], got_s.ravel(), ref["col_scale"].ravel())
            assert nd <= max(1, 1e-4 * got_d.size * 2), f"{nd} RHT code differences"
    return ref


def test_1d_1024x1024_full(oracle_mod):
    spec = inputs.WORKLOADS["1d_1024x1024_bf16"]
    x = inputs.make(spec)
    q = nv.quantize(x.cuda(), "1d", swizzled=False)
    torch.cuda.synchronize()
    ref = oracle_mod.quantize("1d", bits(x))
    from nvfp4_testutil import assert_quantize_equal
    assert_quantize_equal(oracle_mod, q, ref, False)


def test_2d_8192x5120_swizzled_with_dequant(oracle_mod):
    spec = inputs.WORKLOADS["2d_8192x5120_bf16"]
    x = inputs.make(spec)
    xd = x.cuda()
    q = nv.quantize(xd, "2d", swizzled=True)
    y = nv.dequantize(q.data_row, q.scale_row, q.amax_row, swizzled=True)
    torch.cuda.synchronize()
    M, N = x.shape
    rows = _sample(M, 48, 1, must=(0, 15, 16, M - 1))
    cols = _sample(N, 48, 2, must=(0, N - 1))
    ref = _check_sampled(oracle_mod, q, bits(x), "2d", rows, cols, True)
    deq = oracle_mod.dequantize(ref["row_data"], ref["row_scale"], ref["amax_row"], False, "bf16")
    np.testing.assert_array_equal(bits(y)[rows], deq)
    # size-independent: the swizzled scales are the compact ones permuted
    qc = nv.quantize(xd, "2d", swizzled=False)
    assert torch.equal(qc.data_row, q.data_row) and torch.equal(qc.data_col, q.data_col)
    assert torch.equal(nv.swizzle_scales(qc.scale_row, M, N // 16), q.scale_row)
    assert torch.equal(nv.swizzle_scales(qc.scale_col, N, M // 16), q.scale_col)


@pytest.mark.parametrize("swizzled", [False, True])
def test_2d_single_pass_many_tiles_per_cta(oracle_mod, swizzled):
    # 16384x5120: 5120 tiles, 34 per CTA on 152 SMs -- more than the 2D
    # single-pass kernel keeps tile maxima for, so phase B finds them again;
    # most tiles are re-read in phase B
    x = inputs.randn(16384, 5120, seed=11)
    q = nv.quantize(x.cuda(), "2d", swizzled=swizzled, path="single_pass")
    torch.cuda.synchronize()
    xb = bits(x)
    M, N = xb.shape
    assert np_(q.amax_row)[0] == oracle_mod.amax(xb)
    rows = _sample(M, 32, 7, must=(0, 16, M - 1))
    cols = _sample(N, 32, 8, must=(0, N - 1))
    _check_sampled(oracle_mod, q, xb, "2d", rows, cols, swizzled)
    assert nv.device_status() == 0


@pytest.mark.parametrize("swizzled", [False, True])
def test_row_scaled_16384x4096(oracle_mod, swizzled):
    spec = inputs.WORKLOADS["rowscaled_16384x4096_bf16"]
    x = inputs.make(spec)
    q = nv.quantize(x.cuda(), "row_scaled", swizzled=swizzled)
    torch.cuda.synchronize()
    xb = bits(x)
    M, N = xb.shape
    a = np.abs((xb.astype(np.uint32) << 16).view(np.float32)).max(axis=1)
    np.testing.assert_array_equal(np_(q.amax_row), a)                  # every row's amax
    big = np.nonzero(a > 50)[0][:8]
    zero = np.nonzero(a == 0)[0][:8]
    assert big.size > 0 and zero.size > 0
    rows = _sample(M, 160, 3, must=list(big) + list(zero) + [0, M - 1])
    _check_sampled(oracle_mod, q, xb, "row_scaled", rows, None, swizzled)
    assert bool((q.data_row[torch.from_numpy(zero).cuda()] == 0).all())


@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_rht_8192x8192(oracle_mod, path):
    spec = inputs.WORKLOADS["rht_8192x8192_bf16"]
    x = inputs.make(spec)
    mask = inputs.sign_mask_from_seed(spec["seed"])
    q = nv.quantize(x.cuda(), "rht", sign_mask=mask, swizzled=False, path=path)
    torch.cuda.synchronize()
    xb = bits(x)
    assert np_(q.amax_row)[0] == oracle_mod.amax(xb)
    assert np_(q.amax_col)[0] == oracle_mod.rht_amax(xb, mask)
    M, N = xb.shape
    _check_sampled(oracle_mod, q, xb, "rht", _sample(M, 32, 4), _sample(N, 32, 5), False, mask,
                   exact_cols=False)


@pytest.mark.parametrize("name", ["1d_1088x1024_bf16", "1d_4096x3072_fp32", "1d_8192x5120_bf16",
                                  "1d_16384x16384_bf16"])
def test_1d_sweep_with_reuse_sequence(oracle_mod, name):
    spec = inputs.WORKLOADS[name]
    base = inputs.make(spec)
    M, N = base.shape
    swizzled = spec["swizzled"] and M % 128 == 0 and N % 128 == 0
    q = nv.empty(M, N, device="cuda")
    rows = _sample(M, 24, 6, must=(0, M - 1))
    cols = _sample(N, 24, 7, must=(0, N - 1))
    for i, x in enumerate(inputs.reuse_sequence(base)):
        xd = x.cuda()
        nv.quantize(xd, "1d", swizzled=swizzled, out=q)
        torch.cuda.synchronize()
        a = oracle_mod.amax(bits(x))
        assert q.amax_row.item() == a and q.amax_col.item() == a, f"step {i}"
        if i in (0, 3) or M * N <= 4096 * 3072:
            _check_sampled(oracle_mod, q, bits(x), "1d", rows, cols, swizzled)
        del xd
    torch.cuda.empty_cache()
