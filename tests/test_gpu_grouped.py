"""Grouped (multi-tensor) quantize against the oracle, member by member and
bit for bit, through both paths (BF16: the single launch and the three
launches; FP32: the three launches): members of uneven height (ragged
128-row tiles at every member boundary, where a tile also holds the next
member's rows, empty members), magnitudes far apart (so a shared amax, or a
boundary tile's maximum leaking into the wrong member, would show), 1D / 2D,
row / column / both, compact and swizzled scales; then many small members,
noop, skip-amax, reuse of the outputs, single-launch calls interleaved with
other single-pass calls on one workspace, and the grouped workload at full
size compared whole."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import assert_quantize_equal, bits, np_, scales_compact

pytestmark = pytest.mark.gpu

FLAGS = [(True, True), (True, False), (False, True)]


def _spec(dtype):
    return dict(inputs.GROUPED, dtype=dtype)


def _check_members(oracle_mod, outs, refs, swizzled, rowwise, colwise, what):
    assert len(outs) == len(refs)
    for g, (q, ref) in enumerate(zip(outs, refs)):
        assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise, colwise, what=f"{what} member {g}")


def _paths(dtype):
    return ["single_pass", "three_pass"] if dtype == torch.bfloat16 else ["three_pass"]


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
        for path in _paths(dtype):
            outs = nv.quantize_grouped(xd, splits, mode, rowwise=rowwise, colwise=colwise, path=path)
            torch.cuda.synchronize()
            _check_members(oracle_mod, outs, refs, False, rowwise, colwise,
                           f"{mode} {dtype} r{rowwise}c{colwise} {path}")
    assert nv.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_grouped_swizzled_matches_oracle(oracle_mod, dtype, mode):
    splits = [256, 128, 0, 384, 128]
    x = inputs.make_grouped(_spec(dtype), splits=splits, N=384)
    xd = x.cuda()
    for rowwise, colwise in FLAGS:
        refs = oracle_mod.quantize_grouped(mode, bits(x), splits, rowwise=rowwise, colwise=colwise)
        for path in _paths(dtype):
            outs = nv.quantize_grouped(xd, splits, mode, rowwise=rowwise, colwise=colwise, swizzled=True, path=path)
            torch.cuda.synchronize()
            _check_members(oracle_mod, outs, refs, True, rowwise, colwise, f"{mode} {dtype} swizzled {path}")


def test_grouped_row_only_any_member_height(oracle_mod):
    # the row-wise 1D output alone needs no 16-row blocks: any member height
    splits = [40, 1, 87, 0, 128, 5]
    x = inputs.make_grouped(splits=splits, N=96)
    refs = oracle_mod.quantize_grouped("1d", bits(x), splits, colwise=False)
    for path in ("single_pass", "three_pass"):
        outs = nv.quantize_grouped(x.cuda(), splits, "1d", colwise=False, path=path)
        torch.cuda.synchronize()
        _check_members(oracle_mod, outs, refs, False, True, False, f"row-only {path}")


def test_grouped_sixty_four_members(oracle_mod):
    rng = np.random.default_rng(5)
    splits = [int(16 * k) for k in rng.integers(0, 9, size=64)]
    splits[7] = 0
    x = inputs.make_grouped(splits=splits, N=160)
    for mode in ("1d", "2d"):
        refs = oracle_mod.quantize_grouped(mode, bits(x), splits)
        for path in ("single_pass", "three_pass"):
            outs = nv.quantize_grouped(x.cuda(), splits, mode, path=path)
            torch.cuda.synchronize()
            _check_members(oracle_mod, outs, refs, False, True, True, f"64 members {mode} {path}")


def test_grouped_one_member_equals_plain_quantize():
    x = inputs.randn(384, 512, seed=9).cuda()
    for mode in ("1d", "2d"):
        p = nv.quantize(x, mode, swizzled=True, path="two_pass")
        for path in ("single_pass", "three_pass"):
            (g,) = nv.quantize_grouped(x, [384], mode, swizzled=True, path=path)
            torch.cuda.synchronize()
            for a, b in ((g.data_row, p.data_row), (g.scale_row, p.scale_row), (g.amax_row, p.amax_row),
                         (g.data_col, p.data_col), (g.scale_col, p.scale_col), (g.amax_col, p.amax_col)):
                assert torch.equal(a, b), path


def test_grouped_single_pass_shares_the_workspace(oracle_mod):
    """Single-launch grouped calls interleaved, on one workspace, with plain
    single-pass calls (which move the barrier's generation but not the
    members' maxima): every grouped call must still see only its own
    maxima, across both generation parities and a smaller member count."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    big = [256, 128, 384]
    small = [128, 128]
    xa = inputs.make_grouped(dict(inputs.GROUPED, seed=3), splits=big, N=256)
    xb = (inputs.make_grouped(dict(inputs.GROUPED, seed=4), splits=small, N=256).float() * 1e-3).to(torch.bfloat16)
    xp = inputs.randn(256, 512, seed=5)
    ref_a = oracle_mod.quantize_grouped("1d", bits(xa), big)
    ref_b = oracle_mod.quantize_grouped("1d", bits(xb), small)
    ref_p = oracle_mod.quantize("2d", bits(xp))
    plan = ["a", "p", "b", "b", "p", "p", "a", "b", "a", "p", "a"]
    for step, which in enumerate(plan):
        if which == "p":
            q = nv.quantize(xp.cuda(), "2d", path="single_pass", workspace=ws)
            torch.cuda.synchronize()
            assert_quantize_equal(oracle_mod, q, ref_p, False, what=f"plain step {step}")
        else:
            x, splits, refs = (xa, big, ref_a) if which == "a" else (xb, small, ref_b)
            outs = nv.quantize_grouped(x.cuda(), splits, "1d", path="single_pass", workspace=ws)
            torch.cuda.synchronize()
            _check_members(oracle_mod, outs, refs, False, True, True, f"grouped {which} step {step}")
    assert nv.device_status() == 0


def test_grouped_reuse_noop_and_skip_amax(oracle_mod):
    splits = [128, 64, 192]
    base = inputs.make_grouped(splits=splits, N=256)
    outs = [nv.empty(m, 256, device="cuda") for m in splits]
    # the dual-amax reuse sequence, one member zeroed in the last step
    seq = inputs.reuse_sequence(base)
    seq[-1][128:192] = 0
    for it, x in enumerate(seq):
        for path in ("single_pass", "three_pass"):
            nv.quantize_grouped(x.cuda(), splits, "1d", out=outs, path=path)
            torch.cuda.synchronize()
            _check_members(oracle_mod, outs, oracle_mod.quantize_grouped("1d", bits(x), splits), False, True, True,
                           f"reuse step {it} {path}")
    # noop = 1: nothing written
    for q in outs:
        for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
            t.fill_(0xAB)
        q.amax_row.fill_(-3.0)
        q.amax_col.fill_(-3.0)
    noop = torch.ones(1, device="cuda")
    for path in ("single_pass", "three_pass"):
        nv.quantize_grouped(base.cuda(), splits, "2d", out=outs, noop=noop, path=path)
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
    with pytest.raises(ValueError):
        nv.quantize_grouped(x.float(), [32, 32], path="single_pass")       # single launch: bfloat16
    with pytest.raises(ValueError):
        nv.quantize_grouped(x, [32, 32], path="single_pass", skip_amax=True)


@pytest.mark.slow
def test_grouped_full_size_whole(oracle_mod):
    """The grouped workload as the benchmark runs it (the single launch), and
    the three launches: every member's amax, codes and scales (read back
    from the 128x4 layout through the oracle's permutation) compared with one
    oracle call per member, over the whole member."""
    spec = inputs.GROUPED
    splits = spec["splits"]
    x = inputs.make_grouped(spec)
    xb = bits(x)
    N = spec["N"]
    refs, r = [], 0
    for m in splits:
        refs.append(oracle_mod.quantize(spec["mode"], xb[r:r + m]))
        r += m
    xd = x.cuda()
    for path in ("single_pass", "three_pass"):
        outs = nv.quantize_grouped(xd, splits, spec["mode"], swizzled=spec["swizzled"], path=path)
        torch.cuda.synchronize()
        for g, (q, m, ref) in enumerate(zip(outs, splits, refs)):
            what = f"{path} member {g}"
            np.testing.assert_array_equal(np_(q.amax_row), ref["amax_row"], err_msg=what)
            np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"], err_msg=what)
            np.testing.assert_array_equal(np_(q.data_row), ref["row_data"], err_msg=f"{what} row codes")
            np.testing.assert_array_equal(np_(q.data_col), ref["col_data"], err_msg=f"{what} column codes")
            np.testing.assert_array_equal(scales_compact(oracle_mod, np_(q.scale_row), m, N // 16, spec["swizzled"]),
                                          ref["row_scale"], err_msg=f"{what} row scales")
            np.testing.assert_array_equal(scales_compact(oracle_mod, np_(q.scale_col), N, m // 16, spec["swizzled"]),
                                          ref["col_scale"], err_msg=f"{what} column scales")
    assert nv.device_status() == 0
