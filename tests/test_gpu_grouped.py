"""Grouped (multi-tensor) quantize against the oracle, member by member and
bit for bit: members of uneven height (ragged 128-row tiles at every member
boundary, empty members), magnitudes far apart (so a shared amax would show),
1D / 2D, BF16 / FP32, row / column / both, compact and swizzled scales; then
many small members, noop, skip-amax, reuse of the outputs, and the grouped
workload at full size on sampled rows and columns."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import assert_quantize_equal, bits, np_

pytestmark = pytest.mark.gpu

FLAGS = [(True, True), (True, False), (False, True)]


def _spec(dtype):
    return dict(inputs.GROUPED, dtype=dtype)


def _check_members(oracle_mod, outs, refs, swizzled, rowwise, colwise, what):
    assert len(outs) == len(refs)
    for g, (q, ref) in enumerate(zip(outs, refs)):
        assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise, colwise, what=f"{what} member {g}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_grouped_compact_matches_oracle(oracle_mod, dtype, mode):
    # member boundaries inside 128-row tiles, an empty member, N not a
    # multiple of 128 (ragged column tiles)
    splits = [128, 48, 0, 256, 16, 208]
    x = inputs.make_grouped(_spec(dtype), splits=splits, N=336)
    xd = x.cuda()
    for rowwise, colwise in FLAGS:
        refs = oracle_mod.quantize_grouped(mode, bits(x), splits, rowwise=rowwise, colwise=colwise)
        outs = nv.quantize_grouped(xd, splits, mode, rowwise=rowwise, colwise=colwise)
        torch.cuda.synchronize()
        _check_members(oracle_mod, outs, refs, False, rowwise, colwise, f"{mode} {dtype} r{rowwise}c{colwise}")
    assert nv.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_grouped_swizzled_matches_oracle(oracle_mod, dtype, mode):
    splits = [256, 128, 0, 384, 128]
    x = inputs.make_grouped(_spec(dtype), splits=splits, N=384)
    xd = x.cuda()
    for rowwise, colwise in FLAGS:
        refs = oracle_mod.quantize_grouped(mode, bits(x), splits, rowwise=rowwise, colwise=colwise)
        outs = nv.quantize_grouped(xd, splits, mode, rowwise=rowwise, colwise=colwise, swizzled=True)
        torch.cuda.synchronize()
        _check_members(oracle_mod, outs, refs, True, rowwise, colwise, f"{mode} {dtype} swizzled")


def test_grouped_row_only_any_member_height(oracle_mod):
    # the row-wise 1D output alone needs no 16-row blocks: any member height
    splits = [40, 1, 87, 0, 128, 5]
    x = inputs.make_grouped(splits=splits, N=96)
    refs = oracle_mod.quantize_grouped("1d", bits(x), splits, colwise=False)
    outs = nv.quantize_grouped(x.cuda(), splits, "1d", colwise=False)
    torch.cuda.synchronize()
    _check_members(oracle_mod, outs, refs, False, True, False, "row-only")


def test_grouped_sixty_four_members(oracle_mod):
    rng = np.random.default_rng(5)
    splits = [int(16 * k) for k in rng.integers(0, 9, size=64)]
    splits[7] = 0
    x = inputs.make_grouped(splits=splits, N=160)
    for mode in ("1d", "2d"):
        refs = oracle_mod.quantize_grouped(mode, bits(x), splits)
        outs = nv.quantize_grouped(x.cuda(), splits, mode)
        torch.cuda.synchronize()
        _check_members(oracle_mod, outs, refs, False, True, True, f"64 members {mode}")


def test_grouped_one_member_equals_plain_quantize():
    x = inputs.randn(384, 512, seed=9).cuda()
    for mode in ("1d", "2d"):
        (g,) = nv.quantize_grouped(x, [384], mode, swizzled=True)
        p = nv.quantize(x, mode, swizzled=True, path="two_pass")
        torch.cuda.synchronize()
        for a, b in ((g.data_row, p.data_row), (g.scale_row, p.scale_row), (g.amax_row, p.amax_row),
                     (g.data_col, p.data_col), (g.scale_col, p.scale_col), (g.amax_col, p.amax_col)):
            assert torch.equal(a, b)


def test_grouped_reuse_noop_and_skip_amax(oracle_mod):
    splits = [128, 64, 192]
    base = inputs.make_grouped(splits=splits, N=256)
    outs = [nv.empty(m, 256, device="cuda") for m in splits]
    # the dual-amax reuse sequence, one member zeroed in the last step
    seq = inputs.reuse_sequence(base)
    seq[-1][128:192] = 0
    for it, x in enumerate(seq):
        nv.quantize_grouped(x.cuda(), splits, "1d", out=outs)
        torch.cuda.synchronize()
        _check_members(oracle_mod, outs, oracle_mod.quantize_grouped("1d", bits(x), splits), False, True, True,
                       f"reuse step {it}")
    # noop = 1: nothing written
    for q in outs:
        for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
            t.fill_(0xAB)
        q.amax_row.fill_(-3.0)
        q.amax_col.fill_(-3.0)
    noop = torch.ones(1, device="cuda")
    nv.quantize_grouped(base.cuda(), splits, "2d", out=outs, noop=noop)
    torch.cuda.synchronize()
    for q in outs:
        for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
            assert bool((t == 0xAB).all())
        assert q.amax_row.item() == -3.0 and q.amax_col.item() == -3.0
    # skip-amax: each member's buffers are read, not written
    given = []
    r = 0
    for q, m in zip(outs, splits):
        a = oracle_mod.amax(bits(base[r:r + m]))
        q.amax_row.fill_(2 * a)
        q.amax_col.fill_(3 * a)
        given.append((2 * a, 3 * a))
        r += m
    nv.quantize_grouped(base.cuda(), splits, "2d", out=outs, skip_amax=True)
    torch.cuda.synchronize()
    r = 0
    for g, (q, m) in enumerate(zip(outs, splits)):
        ref = oracle_mod.quantize("2d", bits(base[r:r + m]), amax=given[g])
        assert_quantize_equal(oracle_mod, q, ref, False, what=f"skip-amax member {g}")
        r += m


def test_grouped_rejects_bad_arguments():
    x = torch.zeros(64, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        nv.quantize_grouped(x, [32, 16])                  # rows do not add up
    with pytest.raises(ValueError):
        nv.quantize_grouped(x, [1] * 64 + [0])             # too many members
    with pytest.raises(nv.NVFP4Error):
        nv.quantize_grouped(x, [40, 24])                   # column blocks need 16-row members
    with pytest.raises(nv.NVFP4Error):
        nv.quantize_grouped(x, [32, 32], swizzled=True)    # the 128x4 layout needs 128-row members


@pytest.mark.slow
def test_grouped_full_size_sampled(oracle_mod):
    """The grouped workload as the benchmark runs it: every member's amax
    exactly, sampled rows and columns of every member."""
    spec = inputs.GROUPED
    splits = spec["splits"]
    x = inputs.make_grouped(spec)
    outs = nv.quantize_grouped(x.cuda(), splits, spec["mode"], swizzled=spec["swizzled"])
    torch.cuda.synchronize()
    xb = bits(x)
    N = spec["N"]
    rng = np.random.default_rng(3)
    r = 0
    for g, (q, m) in enumerate(zip(outs, splits)):
        xm = xb[r:r + m]
        a = oracle_mod.amax(xm)
        assert np_(q.amax_row)[0] == a and np_(q.amax_col)[0] == a
        rows = np.unique(np.concatenate([rng.choice(m, 8, replace=False), [0, m - 1]])).astype(np.int64)
        cols = np.unique(np.concatenate([rng.choice(N, 8, replace=False), [0, N - 1]])).astype(np.int64)
        ref = oracle_mod.quantize(spec["mode"], xm, rows=rows, cols=cols)
        np.testing.assert_array_equal(np_(q.data_row)[rows], ref["row_data"], err_msg=f"member {g} rows")
        np.testing.assert_array_equal(np_(q.data_col)[cols], ref["col_data"], err_msg=f"member {g} cols")
        off_r = np.array([[oracle_mod.swizzle_offset(int(i), c, N // 16) for c in range(N // 16)] for i in rows])
        off_c = np.array([[oracle_mod.swizzle_offset(int(j), c, m // 16) for c in range(m // 16)] for j in cols])
        np.testing.assert_array_equal(np_(q.scale_row)[off_r], ref["row_scale"], err_msg=f"member {g} row scales")
        np.testing.assert_array_equal(np_(q.scale_col)[off_c], ref["col_scale"], err_msg=f"member {g} col scales")
        r += m
    assert nv.device_status() == 0
