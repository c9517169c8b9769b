"""Parity of the CUDA path with the oracle, element by element, on seeded
inputs that span several 128x128 tiles and ragged tails: amax (both
buffers), E4M3 scales (compact and swizzled), FP4 codes, for 1D / 2D /
row-scaled / RHT quantization, dequantize and the standalone swizzle; plus
the semantics the pages fix (dual amax refreshed on reuse, noop, skip-amax,
graph capture with stable pointers)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_amax_gb300 as nv
from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import assert_quantize_equal, bits, check_rht_columns, np_
from nvfp4_testutil import scales_compact as _compact

pytestmark = pytest.mark.gpu

SHAPES = [(16, 16), (128, 128), (48, 80), (208, 336), (256, 384), (384, 640), (1088, 1024),
          (16, 4096), (4096, 16), (144, 2064)]  # one row block / one column block / thin ragged
DTYPES = [torch.bfloat16, torch.float32]


def _x(M, N, dtype, seed, kind="randn"):
    if kind == "outliers":
        return inputs.outliers(M, N, seed=seed, frac=0.01, dtype=dtype)
    if kind == "row_mix":
        return inputs.row_mix(M, N, seed=seed, frac=0.05, dtype=dtype)
    return inputs.randn(M, N, seed=seed, dtype=dtype)


def _flags():
    return [(True, True), (True, False), (False, True)]



@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("mode", ["1d", "2d"])
@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_quantize_matches_oracle(oracle_mod, M, N, dtype, mode, path):
    x = _x(M, N, dtype, seed=M * 7 + N, kind="outliers")
    xd = x.cuda()
    swz_ok = M % 128 == 0 and N % 128 == 0
    for rowwise, colwise in _flags():
        ref = oracle_mod.quantize(mode, bits(x), rowwise=rowwise, colwise=colwise)
        for swizzled in ([False, True] if swz_ok else [False]):
            q = nv.quantize(xd, mode, rowwise=rowwise, colwise=colwise, swizzled=swizzled, path=path)
            torch.cuda.synchronize()
            assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise, colwise,
                                  what=f"{mode} {path} {M}x{N} {dtype} r{rowwise}c{colwise}s{swizzled}")


@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_single_pass_workspace_reuse(oracle_mod, mode):
    """The grid barrier's generation counter keeps one workspace valid over
    many calls of different grid sizes (tile counts), and across the
    dual-amax reuse sequence."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for it, (M, N) in enumerate([(128, 128), (1024, 2048), (256, 384), (2048, 2048), (16, 16)] * 3):
        base = _x(M, N, torch.bfloat16, seed=it, kind="outliers")
        for x in inputs.reuse_sequence(base):
            q = nv.quantize(x.cuda(), mode, path="single_pass", workspace=ws)
            torch.cuda.synchronize()
            ref = oracle_mod.quantize(mode, bits(x))
            assert_quantize_equal(oracle_mod, q, ref, False, what=f"{mode} {M}x{N} call {it}")
    w = ws.view(torch.int32).cpu()
    assert int(w[0]) == 15 * 4                  # one generation per call
    assert int(w[2 + (60 & 1)]) == 0            # the next call's arrival count is clear
    assert int(w[4 + (60 & 1)]) == 0            # and so is its maximum
    assert nv.device_status() == 0


@pytest.mark.parametrize("M,N", [(16, 16), (128, 128), (48, 80), (208, 336), (384, 640), (1088, 1024),
                                 (16, 2048), (2048, 16)])
@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_rht_matches_oracle(oracle_mod, M, N, path):
    x = _x(M, N, torch.bfloat16, seed=M + 3 * N, kind="outliers")
    mask = inputs.sign_mask_from_seed(M + N)
    ref = oracle_mod.quantize("rht", bits(x), sign_mask=mask)
    for swizzled in ([False, True] if (M % 128 == 0 and N % 128 == 0) else [False]):
        q = nv.quantize(x.cuda(), "rht", sign_mask=mask, swizzled=swizzled, path=path)
        torch.cuda.synchronize()
        assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise=True, colwise=False, what="rht row")
        np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"])
        c = check_rht_columns(oracle_mod, bits(x), mask, np_(q.data_col),
                              _compact(oracle_mod, np_(q.scale_col), N, M // 16, swizzled), ref)
        assert c["codes_differing"] <= 1e-4 * M * N


def test_rht_single_pass_reuse_and_reloads(oracle_mod):
    """Single-pass Hadamard quantize over repeated calls on one workspace,
    shapes with several tiles per CTA (phase-B reloads of tiles that did not
    stay in shared memory), both amaxes and the dual-amax reuse sequence."""
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    calls = 0
    for it, (M, N) in enumerate([(4096, 4352), (128, 128), (1040, 2064), (2048, 1024)]):
        base = _x(M, N, torch.bfloat16, seed=40 + it, kind="outliers")
        mask = inputs.sign_mask_from_seed(it)
        seq = inputs.reuse_sequence(base) if M * N <= 4 << 20 else [base]
        for x in seq:
            ref = oracle_mod.quantize("rht", bits(x), sign_mask=mask)
            for swizzled in ([False, True] if (M % 128 == 0 and N % 128 == 0) else [False]):
                q = nv.quantize(x.cuda(), "rht", sign_mask=mask, swizzled=swizzled, path="single_pass",
                                workspace=ws)
                torch.cuda.synchronize()
                calls += 1
                assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise=True, colwise=False,
                                      what=f"rht {M}x{N} call {calls}")
                np.testing.assert_array_equal(np_(q.amax_col), ref["amax_col"])
                c = check_rht_columns(oracle_mod, bits(x), mask, np_(q.data_col),
                                      _compact(oracle_mod, np_(q.scale_col), N, M // 16, swizzled), ref)
                assert c["codes_differing"] <= 1e-4 * M * N
    w = ws.view(torch.int32).cpu()
    assert int(w[0]) == calls                       # one generation per call
    assert int(w[2 + (calls & 1)]) == 0             # the next call's arrival count is clear
    assert int(w[4 + (calls & 1)]) == 0 and int(w[6 + (calls & 1)]) == 0   # and both its maxima
    assert nv.device_status() == 0


@pytest.mark.parametrize("M,N", [(16, 16), (40, 64), (128, 128), (300, 4096), (256, 6144), (64, 2048)])
@pytest.mark.parametrize("dtype", DTYPES)
def test_row_scaled_matches_oracle(oracle_mod, M, N, dtype):
    x = _x(M, N, dtype, seed=M + N, kind="row_mix")
    ref = oracle_mod.quantize("row_scaled", bits(x), colwise=False)
    for swizzled in ([False, True] if (M % 128 == 0 and N % 128 == 0) else [False]):
        q = nv.quantize(x.cuda(), "row_scaled", swizzled=swizzled)
        torch.cuda.synchronize()
        assert_quantize_equal(oracle_mod, q, ref, swizzled, rowwise=True, colwise=False, what="row_scaled")


def test_row_only_ragged_rows(oracle_mod):
    # row-wise output alone needs only N % 16 == 0: any number of rows
    for M in (1, 5, 129, 1000):
        x = _x(M, 96, torch.bfloat16, seed=M)
        ref = oracle_mod.quantize("1d", bits(x), colwise=False)
        q = nv.quantize(x.cuda(), "1d", colwise=False)
        assert_quantize_equal(oracle_mod, q, ref, False, colwise=False)
        ref = oracle_mod.quantize("row_scaled", bits(x), colwise=False)
        q = nv.quantize(x.cuda(), "row_scaled")
        assert_quantize_equal(oracle_mod, q, ref, False, colwise=False)


def test_empty_inputs():
    for M, N in ((0, 64), (64, 0), (0, 0)):
        x = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        q = nv.empty(M, N, device="cuda")
        q.amax_row.fill_(5.0)
        q.amax_col.fill_(5.0)
        nv.quantize(x, "1d", out=q)
        torch.cuda.synchronize()
        assert q.amax_row.item() == 0.0 and q.amax_col.item() == 0.0


@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_dual_amax_refreshed_on_reuse(oracle_mod, path):
    """'Write both NVFP4 amax buffers', Changes: one output reused over
    inputs whose maximum decreases, reaches zero and rises again."""
    for mode, dtype, (M, N) in [("1d", torch.bfloat16, (256, 256)), ("2d", torch.float32, (128, 384)),
                                ("1d", torch.bfloat16, (1088, 1024))]:
        base = _x(M, N, dtype, seed=11)
        for rowwise, colwise in _flags():
            q = nv.empty(M, N, rowwise, colwise, device="cuda")
            for x in inputs.reuse_sequence(base) + [base * 0.0]:
                nv.quantize(x.cuda(), mode, rowwise=rowwise, colwise=colwise, out=q, path=path)
                torch.cuda.synchronize()
                a = oracle_mod.amax(bits(x))
                if rowwise:
                    assert q.amax_row.item() == a
                if colwise:
                    assert q.amax_col.item() == a
                ref = oracle_mod.quantize(mode, bits(x), rowwise=rowwise, colwise=colwise)
                assert_quantize_equal(oracle_mod, q, ref, False, rowwise, colwise)


def test_compute_amax_matches_oracle(oracle_mod):
    for (M, N), dtype in [((1, 8), torch.bfloat16), ((3, 5), torch.float32), ((1000, 999), torch.bfloat16),
                          ((4096, 3072), torch.float32), ((8192, 5120), torch.bfloat16)]:
        x = _x(M, N, dtype, seed=M + N, kind="outliers" if M > 8 else "randn")
        a = torch.full((1,), -1.0, device="cuda")
        b = torch.full((1,), -1.0, device="cuda")
        nv.compute_amax(x.cuda(), a, b)
        torch.cuda.synchronize()
        ref = oracle_mod.amax(bits(x))
        assert a.item() == ref and b.item() == ref
        nv.compute_amax(x.cuda(), a)
        assert a.item() == ref


def test_compute_amax_rht_matches_oracle(oracle_mod):
    for M, N in [(16, 16), (64, 128), (1024, 2048)]:
        x = _x(M, N, torch.bfloat16, seed=N, kind="outliers")
        mask = inputs.sign_mask_from_seed(M)
        a = torch.zeros(1, device="cuda")
        b = torch.zeros(1, device="cuda")
        nv.compute_amax_rht(x.cuda(), mask, a, b)
        torch.cuda.synchronize()
        assert a.item() == oracle_mod.amax(bits(x))
        assert b.item() == oracle_mod.rht_amax(bits(x), mask)


@pytest.mark.parametrize("path", ["two_pass", "auto"])
def test_noop_leaves_everything_untouched(path):
    M, N = 256, 256
    x = _x(M, N, torch.bfloat16, seed=2).cuda()
    for mode in ("1d", "2d", "rht", "row_scaled"):
        q = nv.empty(M, N, colwise=mode != "row_scaled", row_scaled=mode == "row_scaled", device="cuda")
        for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
            if t is not None:
                t.fill_(0xAB)
        for t in (q.amax_row, q.amax_col):
            if t is not None:
                t.fill_(-3.0)
        noop = torch.ones(1, device="cuda")
        nv.quantize(x, mode, out=q, noop=noop, sign_mask=0x1234, path=path if mode in ("1d", "2d") else "auto")
        torch.cuda.synchronize()
        for t in (q.data_row, q.scale_row, q.data_col, q.scale_col):
            if t is not None:
                assert bool((t == 0xAB).all())
        for t in (q.amax_row, q.amax_col):
            if t is not None:
                assert bool((t == -3.0).all())
        noop.zero_()
        nv.quantize(x, mode, out=q, noop=noop, sign_mask=0x1234, path=path if mode in ("1d", "2d") else "auto")
        torch.cuda.synchronize()
        assert q.amax_row[0].item() > 0


def test_skip_amax_uses_given_amax(oracle_mod):
    M, N = 256, 384
    x = _x(M, N, torch.bfloat16, seed=4)
    a = oracle_mod.amax(bits(x))
    for mode in ("1d", "2d"):
        q = nv.empty(M, N, device="cuda")
        q.amax_row.fill_(2 * a)
        q.amax_col.fill_(3 * a)
        nv.quantize(x.cuda(), mode, out=q, skip_amax=True)
        torch.cuda.synchronize()
        ref = oracle_mod.quantize(mode, bits(x), amax=(2 * a, 3 * a))
        assert_quantize_equal(oracle_mod, q, ref, False)
    q = nv.empty(M, N, row_scaled=True, colwise=False, device="cuda")
    per_row = torch.full((M,), float(a), device="cuda")
    q.amax_row.copy_(per_row)
    nv.quantize(x.cuda(), "row_scaled", out=q, skip_amax=True)
    ref = oracle_mod.quantize("1d", bits(x), colwise=False, amax=(a, a))
    np.testing.assert_array_equal(np_(q.data_row), ref["row_data"])


@pytest.mark.parametrize("mode,swizzled", [("1d", False), ("2d", True), ("row_scaled", True), ("row_scaled", False)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_dequantize_matches_oracle(oracle_mod, mode, swizzled, out_dtype):
    M, N = 256, 384
    x = _x(M, N, torch.bfloat16, seed=9, kind="row_mix" if mode == "row_scaled" else "outliers")
    q = nv.quantize(x.cuda(), mode, swizzled=swizzled)
    row_scaled = mode == "row_scaled"
    y = nv.dequantize(q.data_row, q.scale_row, q.amax_row, swizzled=swizzled, row_scaled=row_scaled,
                      out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref_q = oracle_mod.quantize(mode, bits(x), colwise=False)
    ref = oracle_mod.dequantize(ref_q["row_data"], ref_q["row_scale"], ref_q["amax_row"], row_scaled,
                                "bf16" if out_dtype == torch.bfloat16 else "fp32")
    np.testing.assert_array_equal(bits(y), ref)
    if not row_scaled:
        yc = nv.dequantize(q.data_col, q.scale_col, q.amax_col, swizzled=swizzled, out_dtype=out_dtype)
        ref_q = oracle_mod.quantize(mode, bits(x), rowwise=False)
        refc = oracle_mod.dequantize(ref_q["col_data"], ref_q["col_scale"], ref_q["amax_col"], False,
                                     "bf16" if out_dtype == torch.bfloat16 else "fp32")
        np.testing.assert_array_equal(bits(yc), refc)


def test_swizzle_kernel_matches_oracle(oracle_mod):
    rng = np.random.default_rng(3)
    for R, C in [(128, 4), (256, 64), (1024, 320)]:
        compact = rng.integers(0, 256, (R, C), dtype=np.uint8)
        out = nv.swizzle_scales(torch.from_numpy(compact).cuda(), R, C)
        np.testing.assert_array_equal(np_(out), oracle_mod.swizzle(compact))


def test_swizzled_is_permutation_of_compact():
    """'Fuse NVFP4 scale swizzling on SM120 and SM121', Tests: fused
    swizzled output == compact output plus an independent permutation."""
    for mode in ("1d", "2d", "rht", "row_scaled"):
        M, N = 512, 768
        x = _x(M, N, torch.bfloat16, seed=5, kind="outliers").cuda()
        a = nv.quantize(x, mode, swizzled=False, sign_mask=0xF0F0)
        b = nv.quantize(x, mode, swizzled=True, sign_mask=0xF0F0)
        for da, db in ((a.data_row, b.data_row), (a.data_col, b.data_col)):
            if da is not None:
                assert torch.equal(da, db)
        for sa, sb, R in ((a.scale_row, b.scale_row, M), (a.scale_col, b.scale_col, N)):
            if sa is not None:
                assert torch.equal(nv.swizzle_scales(sa, R, sa.numel() // R), sb)


def test_cuda_graph_replay_with_stable_pointers(oracle_mod):
    """'Fuse NVFP4 scale swizzling on SM120 and SM121', Description: cached
    weights need stable scale buffers for CUDA graph replay.  The library
    never allocates, so a captured quantize replays into the same buffers."""
    M, N = 512, 640
    x = _x(M, N, torch.bfloat16, seed=6).cuda()
    q = nv.empty(M, N, swizzled=True, device="cuda")
    ptrs = [t.data_ptr() for t in (q.data_row, q.scale_row, q.data_col, q.scale_col)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nv.quantize(x, "2d", swizzled=True, out=q)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nv.quantize(x, "2d", swizzled=True, out=q)
    for scale in (1.0, 0.25, 8.0):
        x.copy_(_x(M, N, torch.bfloat16, seed=6).cuda() * scale)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_mod.quantize("2d", bits(x))
        assert_quantize_equal(oracle_mod, q, ref, True)
    assert ptrs == [t.data_ptr() for t in (q.data_row, q.scale_row, q.data_col, q.scale_col)]


def test_device_status_clean():
    assert nv.device_status(clear=True) == 0


@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_rejected_shape_writes_nothing(path):
    """A column-wise-only call with N % 16 != 0 is rejected on the host
    before anything is enqueued ("Write both NVFP4 amax buffers", Changes:
    a call that must not write leaves both amax buffers untouched): the
    status is NVFP4_ERR_SHAPE and no buffer changes."""
    M, N = 64, 24
    x = _x(M, N, torch.bfloat16, seed=1).cuda()
    q = nv.empty(M, 32, rowwise=False, colwise=True, device="cuda")   # buffers large enough for N = 32
    q.data_col.fill_(0x5A)
    q.scale_col.fill_(0x5A)
    q.amax_col.fill_(-7.0)
    q.N = N
    with pytest.raises(nv.NVFP4Error) as err:
        nv.quantize(x, "1d", rowwise=False, colwise=True, out=q, path=path)
    assert err.value.status == 2
    torch.cuda.synchronize()
    assert q.amax_col.item() == -7.0
    assert bool((q.data_col == 0x5A).all()) and bool((q.scale_col == 0x5A).all())


@pytest.mark.parametrize("mode,path", [("1d", "auto"), ("2d", "auto"), ("rht", "auto"), ("row_scaled", "auto"),
                                       ("2d", "two_pass"), ("rht", "single_pass")])
def test_quantize_plan_matches_quantize(oracle_mod, mode, path):
    """A QuantizePlan, bound once, gives what quantize gives, call after call
    on the same (updated in place) input; on another stream too."""
    M, N = 256, 384
    x = _x(M, N, torch.bfloat16, seed=21, kind="outliers").cuda()
    mask = 0x1357 if mode == "rht" else 0
    plan = nv.QuantizePlan(x, mode, swizzled=True, sign_mask=mask, path=path)
    s = torch.cuda.Stream()
    for i, scale in enumerate((1.0, 0.5, 4.0)):
        x.mul_(scale)                                   # powers of two: exact in BF16
        if i == 2:
            s.wait_stream(torch.cuda.current_stream())
            q = plan(stream=s)
            torch.cuda.current_stream().wait_stream(s)
        else:
            q = plan()
        ref = nv.quantize(x, mode, swizzled=True, sign_mask=mask)
        torch.cuda.synchronize()
        for a, b in ((q.data_row, ref.data_row), (q.scale_row, ref.scale_row), (q.amax_row, ref.amax_row),
                     (q.data_col, ref.data_col), (q.scale_col, ref.scale_col), (q.amax_col, ref.amax_col)):
            if b is not None:
                assert torch.equal(a, b)
        assert_quantize_equal(oracle_mod, q, oracle_mod.quantize(mode, bits(x), colwise=mode != "row_scaled",
                                                                 sign_mask=mask), True,
                              colwise=mode not in ("row_scaled", "rht"))
