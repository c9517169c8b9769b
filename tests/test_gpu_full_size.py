"""Parity at the full workload sizes, in the launch configuration the
benchmark times: every output of every workload compared with the oracle
element by element over the whole tensor -- amax, codes and scales (read
back from the 128x4 layout through the oracle's permutation), the
row-wise and column-wise dequantize of the headline workload -- plus the
size-independent properties (swizzled = permuted compact, the dual-amax
reuse sequence).  The Hadamard workload's column-wise output is held to
the rounding-tie tolerance (check_rht_columns), its counts printed.

Apart from the headline workload, whose oracle is one whole-tensor call,
the oracle runs as slabs of output rows on the host's cores
(oracle_quantize_slabs; the same numbers as one call, checked on the CPU
in test_testutil.py)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import bits, check_rht_columns, np_, oracle_quantize_slabs, scales_compact

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_whole(oracle, q, xb, mode, swizzled, ref, sign_mask=0, what="", cache=None):
    """Every output of q against the oracle's output `ref` for all of x."""
    M, N = xb.shape
    if q.data_row is not None:
        np.testing.assert_array_equal(np_(q.amax_row), ref["amax_row"], err_msg=f"{what} amax_row")
        np.testing.assert_array_equal(np_(q.data_row), ref["row_data"], err_msg=f"{what} row codes")
        np.testing.assert_array_equal(scales_compact(oracle, np_(q.scale_row), M, N // 16, swizzled),
                                      ref["row_scale"], err_msg=f"{what} row scales")
    if q.data_col is not None:
        np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"], err_msg=f"{what} amax_col")
        got_s = scales_compact(oracle, np_(q.scale_col), N, M // 16, swizzled)
        if mode == "rht":
            c = check_rht_columns(oracle, xb, sign_mask, np_(q.data_col), got_s, ref, cache=cache)
            assert c["codes_differing"] <= 1e-4 * M * N, f"{what}: {c}"
            return c
        np.testing.assert_array_equal(np_(q.data_col), ref["col_data"], err_msg=f"{what} column codes")
        np.testing.assert_array_equal(got_s, ref["col_scale"], err_msg=f"{what} column scales")
    return None


def test_1d_1024x1024_full(oracle_mod):
    spec = inputs.WORKLOADS["1d_1024x1024_bf16"]
    x = inputs.make(spec)
    q = nv.quantize(x.cuda(), "1d", swizzled=False)
    torch.cuda.synchronize()
    ref = oracle_mod.quantize("1d", bits(x))
    _check_whole(oracle_mod, q, bits(x), "1d", False, ref, what="1d 1024x1024")


def test_2d_8192x5120_swizzled_with_dequant(oracle_mod):
    spec = inputs.WORKLOADS["2d_8192x5120_bf16"]
    x = inputs.make(spec)
    xd = x.cuda()
    q = nv.quantize(xd, "2d", swizzled=True)
    y = nv.dequantize(q.data_row, q.scale_row, q.amax_row, swizzled=True)
    yc = nv.dequantize(q.data_col, q.scale_col, q.amax_col, swizzled=True)
    torch.cuda.synchronize()
    xb = bits(x)
    M, N = xb.shape
    ref = oracle_mod.quantize("2d", xb)                 # one whole-tensor oracle call
    _check_whole(oracle_mod, q, xb, "2d", True, ref, what="2d 8192x5120")
    deq = oracle_mod.dequantize(ref["row_data"], ref["row_scale"], ref["amax_row"], False, "bf16")
    np.testing.assert_array_equal(bits(y), deq)
    deq_c = oracle_mod.dequantize(ref["col_data"], ref["col_scale"], ref["amax_col"], False, "bf16")
    np.testing.assert_array_equal(bits(yc), deq_c)
    # size-independent: the swizzled scales are the compact ones permuted
    qc = nv.quantize(xd, "2d", swizzled=False)
    assert torch.equal(qc.data_row, q.data_row) and torch.equal(qc.data_col, q.data_col)
    assert torch.equal(nv.swizzle_scales(qc.scale_row, M, N // 16), q.scale_row)
    assert torch.equal(nv.swizzle_scales(qc.scale_col, N, M // 16), q.scale_col)


def test_2d_single_pass_many_tiles_per_cta(oracle_mod):
    # 16384x5120: 5120 tiles, 34 per CTA on 152 SMs -- more than the 2D
    # single-pass kernel keeps tile maxima for, so phase B finds them again;
    # most tiles are re-read in phase B
    x = inputs.randn(16384, 5120, seed=11)
    xb = bits(x)
    ref = oracle_quantize_slabs(oracle_mod, "2d", xb)
    xd = x.cuda()
    for swizzled in (False, True):
        q = nv.quantize(xd, "2d", swizzled=swizzled, path="single_pass")
        torch.cuda.synchronize()
        _check_whole(oracle_mod, q, xb, "2d", swizzled, ref, what=f"2d 16384x5120 swizzled={swizzled}")
    assert nv.device_status() == 0


def test_row_scaled_16384x4096(oracle_mod):
    spec = inputs.WORKLOADS["rowscaled_16384x4096_bf16"]
    x = inputs.make(spec)
    xb = bits(x)
    ref = oracle_quantize_slabs(oracle_mod, "row_scaled", xb, colwise=False)
    a = ref["amax_row"]
    assert (a > 50).sum() > 0 and (a == 0).sum() > 0      # the workload's x100 rows and zero rows
    xd = x.cuda()
    for swizzled in (False, True):
        q = nv.quantize(xd, "row_scaled", swizzled=swizzled)
        torch.cuda.synchronize()
        _check_whole(oracle_mod, q, xb, "row_scaled", swizzled, ref, what=f"row-scaled swizzled={swizzled}")
        zero = torch.from_numpy(np.nonzero(a == 0)[0]).cuda()
        assert bool((q.data_row[zero] == 0).all())


def test_rht_8192x8192(oracle_mod):
    spec = inputs.WORKLOADS["rht_8192x8192_bf16"]
    x = inputs.make(spec)
    mask = inputs.sign_mask_from_seed(spec["seed"])
    xb = bits(x)
    ref = oracle_quantize_slabs(oracle_mod, "rht", xb, sign_mask=mask)
    assert ref["amax_col"][0] == oracle_mod.rht_amax(xb, mask)
    xd = x.cuda()
    ties = {}
    for path in ("two_pass", "single_pass"):
        for swizzled in (False, True):
            q = nv.quantize(xd, "rht", sign_mask=mask, swizzled=swizzled, path=path)
            torch.cuda.synchronize()
            c = _check_whole(oracle_mod, q, xb, "rht", swizzled, ref, sign_mask=mask,
                             what=f"rht 8192x8192 {path} swizzled={swizzled}", cache=ties)
            print(f"rht 8192x8192 {path} swizzled={swizzled}: {c}")


@pytest.mark.parametrize("name", ["1d_1088x1024_bf16", "1d_4096x3072_fp32", "1d_8192x5120_bf16",
                                  "1d_16384x16384_bf16"])
def test_1d_sweep_with_reuse_sequence(oracle_mod, name):
    spec = inputs.WORKLOADS[name]
    base = inputs.make(spec)
    M, N = base.shape
    swizzled = spec["swizzled"] and M % 128 == 0 and N % 128 == 0
    q = nv.empty(M, N, swizzled=swizzled, device="cuda")
    big = M * N > 8192 * 5120
    for i, x in enumerate(inputs.reuse_sequence(base)):
        xd = x.cuda()
        nv.quantize(xd, "1d", swizzled=swizzled, out=q)
        torch.cuda.synchronize()
        xb = bits(x)
        a = oracle_mod.amax(xb)
        assert q.amax_row.item() == a and q.amax_col.item() == a, f"step {i}"
        if big and i in (1, 2):
            # 16384^2: the whole-tensor comparison on the first and last
            # inputs; the zero input must give zero codes and scales
            if i == 2:
                for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
                    assert int(torch.count_nonzero(t)) == 0
            continue
        ref = oracle_quantize_slabs(oracle_mod, "1d", xb)
        _check_whole(oracle_mod, q, xb, "1d", swizzled, ref, what=f"{name} step {i}")
        del xd
    torch.cuda.empty_cache()
