"""Pins of the oracle's quantize / dequantize drivers.

Each check is anchored outside the oracle: closed forms (exact round trips on
constructed inputs, scale invariance, the block holding the tensor maximum
getting scale 448), invariants the pages fix (both amaxes equal max|x|; the
column-wise output is the quantization of x transposed; row-scaled rows are
independent tensors; RHT amaxes), an error bound, and brute force on small
inputs by a vectorised numpy restatement whose rounding steps are library
routines (numpy round-half-even, PyTorch FP8/BF16 casts).
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_amax_gb300 import inputs

FLT_MAX = np.float32(np.finfo(np.float32).max)
E2M1_GRID = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f32(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.float32)


# ---------------------------------------------------------------------------
# numpy restatement with library rounding
# ---------------------------------------------------------------------------

def np_e2m1(v):
    m = np.abs(v.astype(np.float64))
    val = np.where(m < 2.0, np.rint(m * 2.0) / 2.0,
                   np.where(m < 4.0, np.rint(m), np.where(m < 6.0, 2.0 * np.rint(m / 2.0), 6.0)))
    code = np.searchsorted(E2M1_GRID, val).astype(np.uint8)
    return code | np.where(np.signbit(v), 8, 0).astype(np.uint8)


def np_e4m3(v):
    sat = v > 448.0
    c = torch.from_numpy(np.where(sat, 0, v).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.where(sat, 0x7E, c).astype(np.uint8)


def np_e4m3_value(c):
    return torch.from_numpy(c.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def np_global(a):
    a = np.float32(a)
    if a == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore", divide="ignore"):
        g = np.float32(2688.0) / a
    return FLT_MAX if np.isinf(g) else g


def np_rows_from_block_amax(X, b, g):
    """Codes and scales of rows X (R x C) given per-block maxima b (R x C/16)
    and per-row global scales g (R)."""
    g = np.asarray(g, np.float32).reshape(-1, 1)
    sf = (b / np.float32(6.0)) * g
    s = np_e4m3(sf)
    sv = np_e4m3_value(s)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.where(s == 0, np.float32(0), np.minimum(g / sv, FLT_MAX)).astype(np.float32)
    p = X * np.repeat(r, 16, axis=1)
    q = np_e2m1(p)
    data = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return data, s


def np_quantize_1d_rows(X, g):
    R, C = X.shape
    b = np.abs(X).reshape(R, C // 16, 16).max(-1)
    return np_rows_from_block_amax(X, b, g)


def np_quantize_2d_rows(X, g):
    R, C = X.shape
    t = np.abs(X).reshape(R // 16, 16, C // 16, 16).max(axis=(1, 3))
    b = np.repeat(t, 16, axis=0)
    return np_rows_from_block_amax(X, b, np.full(R, g, np.float32))


def np_rht_columns(X, mask, round_bf16):
    """x^T after the column-block RHT, via an FP64 matrix product (exact for
    the small-integer-scaled inputs used with it) rounded once to FP32."""
    from oracle import hadamard16
    H = hadamard16().astype(np.float64)
    M, N = X.shape
    sign = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    blocks = X.astype(np.float64).reshape(M // 16, 16, N) * sign[None, :, None]
    t = np.einsum("oi,kin->kon", H, blocks) / 4.0
    t = t.reshape(M, N).T.astype(np.float32)
    if round_bf16:
        t = torch.from_numpy(np.ascontiguousarray(t)).to(torch.bfloat16).float().numpy()
    return np.ascontiguousarray(t)


def nibble_transpose(data, rows, cols):
    q = np.empty((rows, cols), np.uint8)
    q[:, 0::2] = data & 0xF
    q[:, 1::2] = data >> 4
    qt = np.ascontiguousarray(q.T)
    return (qt[:, 0::2] | (qt[:, 1::2] << 4)).astype(np.uint8)


# ---------------------------------------------------------------------------
# brute force against the restatement
# ---------------------------------------------------------------------------

SHAPES = [(16, 16), (32, 48), (64, 128), (48, 80), (128, 256)]


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_1d_matches_restatement(oracle_mod, M, N, dtype):
    xt = inputs.randn(M, N, seed=M + N, dtype=dtype)
    x = bf16_bits(xt) if dtype == torch.bfloat16 else xt.numpy()
    X = to_f32(x)
    out = oracle_mod.quantize("1d", x)
    a = np.abs(X).max()
    assert out["amax_row"][0] == a and out["amax_col"][0] == a
    g = np_global(a)
    d, s = np_quantize_1d_rows(X, np.full(M, g, np.float32))
    np.testing.assert_array_equal(out["row_data"], d)
    np.testing.assert_array_equal(out["row_scale"], s)
    dT, sT = np_quantize_1d_rows(np.ascontiguousarray(X.T), np.full(N, g, np.float32))
    np.testing.assert_array_equal(out["col_data"], dT)
    np.testing.assert_array_equal(out["col_scale"], sT)


@pytest.mark.parametrize("M,N", SHAPES)
def test_2d_matches_restatement(oracle_mod, M, N):
    x = bf16_bits(inputs.randn(M, N, seed=3 * M + N))
    X = to_f32(x)
    out = oracle_mod.quantize("2d", x)
    g = np_global(np.abs(X).max())
    d, s = np_quantize_2d_rows(X, g)
    np.testing.assert_array_equal(out["row_data"], d)
    np.testing.assert_array_equal(out["row_scale"], s)
    # column-wise: the nibble transpose of the row-wise codes, transposed scales
    np.testing.assert_array_equal(out["col_data"], nibble_transpose(out["row_data"], M, N))
    np.testing.assert_array_equal(out["col_scale"], np.repeat(s[::16, :].T, 16, axis=0))


@pytest.mark.parametrize("M,N", [(16, 32), (40, 64), (96, 160)])
def test_row_scaled_matches_restatement(oracle_mod, M, N):
    x = bf16_bits(inputs.row_mix(M, N, seed=M, frac=0.1))
    X = to_f32(x)
    out = oracle_mod.quantize("row_scaled", x, colwise=False)
    a = np.abs(X).max(axis=1)
    np.testing.assert_array_equal(out["amax_row"], a)
    g = np.array([np_global(v) for v in a], np.float32)
    d, s = np_quantize_1d_rows(X, g)
    np.testing.assert_array_equal(out["row_data"], d)
    np.testing.assert_array_equal(out["row_scale"], s)
    # each row is its own tensor: row y equals the per-tensor path on x[y]
    for y in range(0, M, 7):
        one = oracle_mod.quantize("1d", x[y:y + 1], colwise=False)
        np.testing.assert_array_equal(out["row_data"][y], one["row_data"][0])
        np.testing.assert_array_equal(out["row_scale"][y], one["row_scale"][0])
    zero_rows = np.where(a == 0)[0]
    assert zero_rows.size > 0
    assert np.all(out["row_data"][zero_rows] == 0) and np.all(out["row_scale"][zero_rows] == 0)


@pytest.mark.parametrize("M,N,mask", [(16, 16, 0), (32, 48, 0xBEEF), (64, 64, 0x1234)])
def test_rht_matches_restatement(oracle_mod, M, N, mask):
    # small integers times 2^-3: every Hadamard sum is exact in FP32, so the
    # FP64 product is the same number
    rng = np.random.default_rng(M * N)
    Xf = (rng.integers(-40, 41, (M, N)) / 8.0).astype(np.float32)
    x = bf16_bits(torch.from_numpy(Xf).to(torch.bfloat16))
    X = to_f32(x)
    out = oracle_mod.quantize("rht", x, sign_mask=mask)
    a_row = np.abs(X).max()
    T = np_rht_columns(X, mask, round_bf16=True)
    a_col = np.abs(T).max()
    assert out["amax_row"][0] == a_row and out["amax_col"][0] == a_col
    d, s = np_quantize_1d_rows(X, np.full(M, np_global(a_row), np.float32))
    np.testing.assert_array_equal(out["row_data"], d)
    np.testing.assert_array_equal(out["row_scale"], s)
    dT, sT = np_quantize_1d_rows(T, np.full(N, np_global(a_col), np.float32))
    np.testing.assert_array_equal(out["col_data"], dT)
    np.testing.assert_array_equal(out["col_scale"], sT)


@pytest.mark.parametrize("M,N,mask", [(16, 16, 0), (32, 48, 0xBEEF), (64, 64, 0x1234)])
def test_rht_columns_match_restatement_when_exact(oracle_mod, M, N, mask):
    # small integers times 2^-3: every Hadamard sum is exact in FP32, so the
    # values before and after the BF16 rounding are the FP64 product's
    rng = np.random.default_rng(M + N + mask)
    Xf = (rng.integers(-40, 41, (M, N)) / 8.0).astype(np.float32)
    x = bf16_bits(torch.from_numpy(Xf).to(torch.bfloat16))
    X = to_f32(x)
    np.testing.assert_array_equal(oracle_mod.rht_columns(x, mask, False), np_rht_columns(X, mask, False))
    np.testing.assert_array_equal(oracle_mod.rht_columns(x, mask, True), np_rht_columns(X, mask, True))
    cols = np.array([N - 1, 0, N // 2])
    np.testing.assert_array_equal(oracle_mod.rht_columns(x, mask, True, cols),
                                  np_rht_columns(X, mask, True)[cols])


@pytest.mark.parametrize("M,N,mask", [(64, 48, 0x5A5A), (256, 32, 0xFFFF)])
def test_rht_columns_on_random_data(oracle_mod, M, N, mask):
    """BF16 values whose exponents spread over 2^-20..2^11, so that many FP32
    Hadamard sums round: they stay within the bound of a 16-term FP32
    summation (15 u sum|terms|, u = 2^-24) of the exact transform; the
    rounded values are the BF16 rounding (PyTorch's cast) of the FP32 sums;
    their maximum is the column amax, and the column-wise output is the 1D
    quantization of the rounded columns."""
    rng = np.random.default_rng(M * N)
    Xf = (rng.standard_normal((M, N)) * 2.0 ** rng.integers(-20, 12, (M, N))).astype(np.float32)
    x = bf16_bits(torch.from_numpy(Xf).to(torch.bfloat16))
    X = to_f32(x)
    t32 = oracle_mod.rht_columns(x, mask, False)
    t16 = oracle_mod.rht_columns(x, mask, True)
    from oracle import hadamard16
    sign = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
    u = X.astype(np.float64).reshape(M // 16, 16, N) * sign[None, :, None]
    exact = (np.einsum("oi,kin->kon", hadamard16().astype(np.float64), u) / 4.0).reshape(M, N).T
    bound = 15 * 2.0 ** -24 * np.repeat(np.abs(u).sum(axis=1) / 4.0, 16, axis=0).T
    assert np.all(np.abs(t32.astype(np.float64) - exact) <= bound)
    assert np.any(t32.astype(np.float64) != exact)           # the case is not trivially exact
    np.testing.assert_array_equal(t16, torch.from_numpy(t32).to(torch.bfloat16).float().numpy())
    assert np.abs(t16).max() == oracle_mod.rht_amax(x, mask)
    out = oracle_mod.quantize("rht", x, sign_mask=mask)
    dT, sT = np_quantize_1d_rows(t16, np.full(N, np_global(np.abs(t16).max()), np.float32))
    np.testing.assert_array_equal(out["col_data"], dT)
    np.testing.assert_array_equal(out["col_scale"], sT)


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def _constructed(rng, M, N, k):
    """x = v * S * 2^k with v on the E2M1 grid (block max |v| = 6) and S an
    E4M3 value per block; one block holds 6 * 448 * 2^k, so amax = 2688 * 2^k
    and g = 2^-k exactly."""
    S_codes = rng.integers(0x08, 0x7E, (M, N // 16)).astype(np.uint8)
    S_codes[0, 0] = 0x7E
    S = np_e4m3_value(S_codes).astype(np.float64)
    q = rng.integers(0, 16, (M, N)).astype(np.uint8)
    q[:, ::16] = 7 | (q[:, ::16] & 8)                   # each block reaches |v| = 6
    v = np.where(q & 8, -1.0, 1.0) * E2M1_GRID[q & 7]
    x = (v * np.repeat(S, 16, axis=1) * 2.0 ** k).astype(np.float32)
    return x, q, S_codes


@pytest.mark.parametrize("k", [-20, 0, 5])
def test_exact_round_trip_on_constructed_input(oracle_mod, k):
    rng = np.random.default_rng(k + 50)
    M, N = 32, 64
    x, q, S_codes = _constructed(rng, M, N, k)
    out = oracle_mod.quantize("1d", x, colwise=False)
    assert out["amax_row"][0] == np.float32(2688.0 * 2.0 ** k)
    np.testing.assert_array_equal(out["row_scale"], S_codes)
    codes = np.empty((M, N), np.uint8)
    codes[:, 0::2] = out["row_data"] & 0xF
    codes[:, 1::2] = out["row_data"] >> 4
    # -0 encodes as +0 only if v was +0; compare values, then signs of nonzeros
    np.testing.assert_array_equal(codes & 7, q & 7)
    nz = (q & 7) != 0
    np.testing.assert_array_equal(codes[nz] & 8, q[nz] & 8)
    back = oracle_mod.dequantize(out["row_data"], out["row_scale"], out["amax_row"], False, "fp32")
    np.testing.assert_array_equal(back, x)


def test_block_holding_the_maximum_gets_scale_448(oracle_mod):
    rng = np.random.default_rng(1)
    for _ in range(2000):
        a = np.float32(np.exp(rng.uniform(np.log(1e-30), np.log(1e30))))
        assert oracle_mod.block_scale(a, oracle_mod.global_encode_scale(a)) == 0x7E


def test_block_scale_divides_by_6_before_multiplying(oracle_mod):
    """Reading of the scale formula block_amax / 6 * global_enc: the FP32
    quotient first, then the product.  Random inputs rarely tell the two FP32
    orders apart, so the cases are built next to E4M3 rounding midpoints
    (block maxima a few ulps around 6*m/g) and kept where (b/6)*g and (b*g)/6
    round to different scales; numpy FP32 arithmetic and PyTorch's E4M3 cast
    give the expected scale."""
    rng = np.random.default_rng(12)
    codes = np.arange(0x08, 0x7E, dtype=np.uint8)
    lo, hi = np_e4m3_value(codes), np_e4m3_value(codes + 1)
    mid = ((lo.astype(np.float64) + hi) / 2)
    g = (np.float32(2688.0) / rng.uniform(0.1, 100.0, mid.size * 64).astype(np.float32)).astype(np.float32)
    m = np.repeat(mid, 64)
    b0 = (6.0 * m / g.astype(np.float64)).astype(np.float32)
    cases = []
    for d in range(-3, 4):
        b = (b0.view(np.int32) + d).view(np.float32)
        first = np_e4m3((b / np.float32(6.0)) * g)
        other = np_e4m3((b * g) / np.float32(6.0))
        sel = np.nonzero(first != other)[0]
        cases += [(b[i], g[i], first[i]) for i in sel]
    assert len(cases) >= 50
    for b, g_, s in cases[:400]:
        assert oracle_mod.block_scale(float(b), float(g_)) == s


def test_global_scale_closed_forms(oracle_mod):
    assert oracle_mod.global_encode_scale(0.0) == 1.0
    assert oracle_mod.global_encode_scale(2688.0) == 1.0
    assert oracle_mod.global_encode_scale(1.0) == 2688.0
    assert oracle_mod.global_encode_scale(1e-40) == float(FLT_MAX)
    assert oracle_mod.encode_factor(0, 5.0) == 0.0
    assert oracle_mod.encode_factor(0x38, 5.0) == 5.0          # s = 1.0
    assert oracle_mod.encode_factor(0x01, 3.0e38) == float(FLT_MAX)


@pytest.mark.parametrize("mode", ["1d", "2d"])
def test_power_of_two_scaling_invariance(oracle_mod, mode):
    X = inputs.randn(64, 96, seed=8, dtype=torch.float32).numpy()
    base = oracle_mod.quantize(mode, X)
    for k in (-12, 3, 40):
        out = oracle_mod.quantize(mode, (X * np.float32(2.0 ** k)).astype(np.float32))
        for key in ("row_data", "row_scale", "col_data", "col_scale"):
            np.testing.assert_array_equal(out[key], base[key])
        assert out["amax_row"][0] == base["amax_row"][0] * np.float32(2.0 ** k)


@pytest.mark.parametrize("mode", ["1d", "2d", "row_scaled"])
def test_dequantize_error_bound(oracle_mod, mode):
    M, N = 64, 128
    x = bf16_bits(inputs.row_mix(M, N, seed=21, frac=0.05)) if mode == "row_scaled" else \
        bf16_bits(inputs.randn(M, N, seed=22))
    X = to_f32(x).astype(np.float64)
    out = oracle_mod.quantize(mode, x, colwise=False)
    back = oracle_mod.dequantize(out["row_data"], out["row_scale"], out["amax_row"], mode == "row_scaled", "fp32")
    a = out["amax_row"].astype(np.float64).reshape(-1, 1) if mode == "row_scaled" else out["amax_row"][0]
    unit = np.repeat(np_e4m3_value(out["row_scale"]).astype(np.float64), 16, axis=1) * (a / 2688.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        m = np.where(unit > 0, np.abs(X) / unit, 0.0)
    half_step = np.where(m < 2, 0.25, np.where(m < 4, 0.5, 1.0)) * unit
    over = np.maximum(np.abs(X) - 6.0 * unit, 0.0)
    bound = np.maximum(half_step, over) * (1 + 1e-6) + 1e-30
    assert np.all(np.abs(back - X) <= bound)
    # the bound is tight enough to notice a wrong 448 / 6 / 2688 constant
    assert np.abs(back - X).max() > 0


def test_dequantize_rounding_and_zero(oracle_mod):
    data = np.array([[0x21, 0x87, 0x00, 0x00, 0xF9, 0x00, 0x00, 0x00]], np.uint8)
    scale = np.array([[0x38]], np.uint8)                       # s = 1.0
    out = oracle_mod.dequantize(data, scale, np.array([2688.0], np.float32), False, "fp32")
    assert list(out[0, :4]) == [0.5, 1.0, 6.0, -0.0]
    assert out[0, 8] == -0.5 and out[0, 9] == -6.0
    zero = oracle_mod.dequantize(data, scale, np.array([0.0], np.float32), False, "bf16")
    assert np.all((zero & 0x7FFF) == 0)


def test_row_scaled_dequant_uses_row_amax(oracle_mod):
    rng = np.random.default_rng(2)
    rows = []
    for y in range(8):
        x, _, _ = _constructed(rng, 1, 32, k=y - 3)
        rows.append(x[0])
    X = np.stack(rows)
    out = oracle_mod.quantize("row_scaled", X, colwise=False)
    np.testing.assert_array_equal(out["amax_row"], np.float32(2688.0) * (2.0 ** (np.arange(8) - 3)).astype(np.float32))
    back = oracle_mod.dequantize(out["row_data"], out["row_scale"], out["amax_row"], True, "fp32")
    np.testing.assert_array_equal(back, X)


def test_column_output_is_row_output_of_transpose(oracle_mod):
    x = bf16_bits(inputs.randn(48, 80, seed=31))
    full = oracle_mod.quantize("1d", x)
    tr = oracle_mod.quantize("1d", np.ascontiguousarray(x.T), colwise=False)
    np.testing.assert_array_equal(full["col_data"], tr["row_data"])
    np.testing.assert_array_equal(full["col_scale"], tr["row_scale"])


def test_selected_rows_and_columns_match_full(oracle_mod):
    x = bf16_bits(inputs.outliers(64, 96, seed=5, frac=0.01))
    rows = np.array([63, 0, 17, 40])
    cols = np.array([95, 3, 50])
    for mode in ("1d", "2d", "rht"):
        full = oracle_mod.quantize(mode, x, sign_mask=0x5A5A)
        part = oracle_mod.quantize(mode, x, sign_mask=0x5A5A, rows=rows, cols=cols)
        np.testing.assert_array_equal(part["row_data"], full["row_data"][rows])
        np.testing.assert_array_equal(part["row_scale"], full["row_scale"][rows])
        np.testing.assert_array_equal(part["col_data"], full["col_data"][cols])
        np.testing.assert_array_equal(part["col_scale"], full["col_scale"][cols])
    rs_full = oracle_mod.quantize("row_scaled", x, colwise=False)
    rs = oracle_mod.quantize("row_scaled", x, colwise=False, rows=rows)
    np.testing.assert_array_equal(rs["row_data"], rs_full["row_data"][rows])
    np.testing.assert_array_equal(rs["amax_row"], rs_full["amax_row"][rows])


def test_given_amax_is_used(oracle_mod):
    x = bf16_bits(inputs.randn(32, 32, seed=1))
    a = oracle_mod.amax(x)
    same = oracle_mod.quantize("1d", x, amax=(a, a))
    ref = oracle_mod.quantize("1d", x)
    for key in ("row_data", "row_scale", "col_data", "col_scale"):
        np.testing.assert_array_equal(same[key], ref[key])
    doubled = oracle_mod.quantize("1d", x, amax=(2 * a, 2 * a))
    assert doubled["amax_row"][0] == 2 * a
    assert not np.array_equal(doubled["row_scale"], ref["row_scale"])


def test_rht_amaxes_follow_the_pages(oracle_mod):
    """Row-wise amax = max|x|, column-wise = max|RHT(x)|, and they differ;
    a single spike of 64 gives row amax 64 and a column amax of about 64/4
    (printed pair: 64 / 16.875 on another program's random draw)."""
    xt = inputs.randn(256, 1024, seed=77)
    x = bf16_bits(xt)
    out = oracle_mod.quantize("rht", x, sign_mask=inputs.sign_mask_from_seed(3))
    assert out["amax_row"][0] == np.abs(to_f32(x)).max()
    assert out["amax_col"][0] != out["amax_row"][0]
    xt[100, 200] = 64.0
    x = bf16_bits(xt)
    out = oracle_mod.quantize("rht", x, sign_mask=inputs.sign_mask_from_seed(3))
    assert out["amax_row"][0] == 64.0
    blk = to_f32(x)[96:112, 200].astype(np.float64)
    rest = (np.abs(blk).sum() - 64.0) / 4.0
    assert abs(out["amax_col"][0] - 16.0) <= rest + 0.125
    assert float(torch.tensor(float(out["amax_col"][0])).to(torch.bfloat16)) == out["amax_col"][0]


def test_shape_domain(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.quantize("1d", np.zeros((16, 24), np.float32))
    with pytest.raises(ValueError):
        oracle_mod.quantize("2d", np.zeros((24, 16), np.float32), colwise=False)
    # row-wise only needs N % 16 == 0; any M
    out = oracle_mod.quantize("1d", np.ones((5, 16), np.float32), colwise=False)
    assert out["row_data"].shape == (5, 8)
    # an empty tensor has amax 0 and no codes
    out = oracle_mod.quantize("1d", np.zeros((0, 32), np.float32), colwise=False)
    assert out["amax_row"][0] == 0.0 and out["row_data"].shape == (0, 16)


# ---------------------------------------------------------------------------
# grouped (multi-tensor) quantize: each member is a tensor of its own
# ---------------------------------------------------------------------------

def test_grouped_members_match_restatement(oracle_mod):
    """Each member against the numpy restatement on its own rows, with the
    amax of its own rows (a member scaled far above the others shows whether
    the amax is shared)."""
    splits = [32, 0, 16, 48]
    x = inputs.randn(sum(splits), 64, seed=41, dtype=torch.float32).numpy()
    x[48:96] *= np.float32(1000.0)
    outs = oracle_mod.quantize_grouped("1d", x, splits)
    assert len(outs) == len(splits)
    r = 0
    for m, out in zip(splits, outs):
        X = x[r:r + m]
        a = np.float32(np.abs(X).max()) if m else np.float32(0)
        assert out["amax_row"][0] == a and out["amax_col"][0] == a
        if m:
            g = np_global(a)
            d, s = np_quantize_1d_rows(X, np.full(m, g, np.float32))
            np.testing.assert_array_equal(out["row_data"], d)
            np.testing.assert_array_equal(out["row_scale"], s)
            dT, sT = np_quantize_1d_rows(np.ascontiguousarray(X.T), np.full(64, g, np.float32))
            np.testing.assert_array_equal(out["col_data"], dT)
            np.testing.assert_array_equal(out["col_scale"], sT)
        else:
            assert out["row_data"].shape == (0, 32) and out["col_data"].shape == (64, 0)
        r += m


def test_grouped_2d_member_matches_restatement(oracle_mod):
    splits = [16, 64]
    x = bf16_bits(inputs.outliers(80, 96, seed=42, frac=0.02))
    outs = oracle_mod.quantize_grouped("2d", x, splits)
    X = to_f32(x)[16:80]
    d, s = np_quantize_2d_rows(X, np_global(np.abs(X).max()))
    np.testing.assert_array_equal(outs[1]["row_data"], d)
    np.testing.assert_array_equal(outs[1]["row_scale"], s)
    np.testing.assert_array_equal(outs[1]["col_data"], nibble_transpose(d, 64, 96))


def test_grouped_single_member_is_the_plain_quantize(oracle_mod):
    x = bf16_bits(inputs.randn(48, 80, seed=43))
    for mode in ("1d", "2d"):
        (one,) = oracle_mod.quantize_grouped(mode, x, [48])
        ref = oracle_mod.quantize(mode, x)
        for key in ("row_data", "row_scale", "amax_row", "col_data", "col_scale", "amax_col"):
            np.testing.assert_array_equal(one[key], ref[key])


def test_grouped_members_are_independent(oracle_mod):
    """Scaling one member by 2^k changes only that member's amax: every code
    and scale of every member stays the same (power-of-two invariance of a
    member that owns its amax)."""
    splits = [16, 32, 16]
    x = inputs.randn(64, 48, seed=44, dtype=torch.float32).numpy()
    base = oracle_mod.quantize_grouped("1d", x, splits)
    y = x.copy()
    y[16:48] *= np.float32(2.0 ** 9)
    moved = oracle_mod.quantize_grouped("1d", y, splits)
    for g, (b, m) in enumerate(zip(base, moved)):
        for key in ("row_data", "row_scale", "col_data", "col_scale"):
            np.testing.assert_array_equal(m[key], b[key])
        factor = np.float32(2.0 ** 9) if g == 1 else np.float32(1.0)
        assert m["amax_row"][0] == b["amax_row"][0] * factor


def test_grouped_rejects_bad_splits(oracle_mod):
    x = np.zeros((32, 16), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.quantize_grouped("1d", x, [16, 8])
    with pytest.raises(ValueError):
        oracle_mod.quantize_grouped("rht", x, [32])


# ---------------------------------------------------------------------------
# stochastic rounding of the codes (random bytes passed in)
# ---------------------------------------------------------------------------

def _rbits(M, N, seed):
    return np.random.default_rng(seed).integers(0, 256, (M, N)).astype(np.uint8)


def np_sr_codes(p, rb):
    """Independent restatement of the stochastic rounding rule on arrays:
    neighbours by searchsorted, f in float64 (exact), up iff rb < 256 f."""
    m = np.abs(p.astype(np.float64))
    sat = m >= 6.0
    lo = np.clip(np.searchsorted(E2M1_GRID, m, side="right") - 1, 0, 6)
    f = (m - E2M1_GRID[lo]) / (E2M1_GRID[lo + 1] - E2M1_GRID[lo])
    code = np.where(sat, 7, lo + (rb.astype(np.float64) < 256.0 * f)).astype(np.uint8)
    return code | np.where(np.signbit(p), 8, 0).astype(np.uint8)


def np_sr_rows(X, b, g, rb):
    g = np.asarray(g, np.float32).reshape(-1, 1)
    s = np_e4m3((b / np.float32(6.0)) * g)
    sv = np_e4m3_value(s)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.where(s == 0, np.float32(0), np.minimum(g / sv, FLT_MAX)).astype(np.float32)
    q = np_sr_codes(X * np.repeat(r, 16, axis=1), rb)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8), s


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_sr_1d_matches_restatement(oracle_mod, dtype):
    M, N = 48, 80
    xt = inputs.outliers(M, N, seed=51, frac=0.02, dtype=dtype)
    x = bits_any(xt)
    X = to_f32(x)
    rb = _rbits(M, N, 52)
    out = oracle_mod.quantize("1d", x, rbits=rb)
    g = np_global(np.abs(X).max())
    b = np.abs(X).reshape(M, N // 16, 16).max(-1)
    d, s = np_sr_rows(X, b, np.full(M, g, np.float32), rb)
    np.testing.assert_array_equal(out["row_data"], d)
    np.testing.assert_array_equal(out["row_scale"], s)
    XT = np.ascontiguousarray(X.T)
    bT = np.abs(XT).reshape(N, M // 16, 16).max(-1)
    dT, sT = np_sr_rows(XT, bT, np.full(N, g, np.float32), np.ascontiguousarray(rb.T))
    np.testing.assert_array_equal(out["col_data"], dT)
    np.testing.assert_array_equal(out["col_scale"], sT)


def bits_any(t):
    return bf16_bits(t) if t.dtype == torch.bfloat16 else t.numpy()


def test_sr_keeps_scales_and_amax(oracle_mod):
    x = bf16_bits(inputs.randn(64, 96, seed=53))
    for mode in ("1d", "2d"):
        rn = oracle_mod.quantize(mode, x)
        sr = oracle_mod.quantize(mode, x, rbits=_rbits(64, 96, 54))
        for key in ("row_scale", "col_scale", "amax_row", "amax_col"):
            np.testing.assert_array_equal(sr[key], rn[key])
        assert (sr["row_data"] != rn["row_data"]).any()


def test_sr_zero_bytes_round_every_product_away_from_zero(oracle_mod):
    x = bf16_bits(inputs.randn(32, 64, seed=55))
    X = to_f32(x)
    out = oracle_mod.quantize("1d", x, colwise=False, rbits=np.zeros((32, 64), np.uint8))
    g = np_global(np.abs(X).max())
    b = np.abs(X).reshape(32, 4, 16).max(-1)
    s = np_e4m3((b / np.float32(6.0)) * g)
    r = np.where(s == 0, np.float32(0), g / np_e4m3_value(s)).astype(np.float32)
    m = np.minimum(np.abs((X * np.repeat(r, 16, axis=1)).astype(np.float64)), 6.0)
    q = np.searchsorted(E2M1_GRID, m, side="left").astype(np.uint8) | np.where(np.signbit(X), 8, 0).astype(np.uint8)
    np.testing.assert_array_equal(out["row_data"], (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))


def test_sr_column_output_uses_the_elements_byte(oracle_mod):
    """Column-wise output of x with bytes rb = row-wise output of x^T with
    bytes rb^T: each element keeps its own random byte in both outputs."""
    x = bf16_bits(inputs.randn(48, 64, seed=56))
    rb = _rbits(48, 64, 57)
    full = oracle_mod.quantize("1d", x, rbits=rb)
    tr = oracle_mod.quantize("1d", np.ascontiguousarray(x.T), colwise=False, rbits=np.ascontiguousarray(rb.T))
    np.testing.assert_array_equal(full["col_data"], tr["row_data"])


def test_sr_2d_columns_are_the_transpose(oracle_mod):
    M, N = 64, 96
    x = bf16_bits(inputs.outliers(M, N, seed=58, frac=0.02))
    out = oracle_mod.quantize("2d", x, rbits=_rbits(M, N, 59))
    np.testing.assert_array_equal(out["col_data"], nibble_transpose(out["row_data"], M, N))


def test_sr_is_unbiased_over_bytes(oracle_mod):
    """Averaged over all 256 bytes, the decoded code of a product p is p to
    within 1/256 of a step (P(up) = ceil(256 f) / 256)."""
    x = np.array([[0.3, -1.1, 2.6, 4.9, 0.02, -5.5, 1.76, 3.14159] * 2], np.float32)
    vals = []
    for byte in range(256):
        out = oracle_mod.quantize("1d", x, colwise=False, rbits=np.full(x.shape, byte, np.uint8))
        q = np.empty(16, np.uint8)
        q[0::2] = out["row_data"][0] & 0xF
        q[1::2] = out["row_data"][0] >> 4
        vals.append(np.where(q & 8, -1.0, 1.0) * E2M1_GRID[q & 7])
    s = out["row_scale"][0, 0]
    g = np_global(np.float32(np.abs(x).max()))
    r = np.float32(g / np_e4m3_value(np.array([s]))[0])
    p = (x[0] * r).astype(np.float64)
    step = np.where(np.abs(p) < 2, 0.5, np.where(np.abs(p) < 4, 1.0, 2.0))
    mean = np.mean(vals, axis=0)
    assert np.all(np.abs(mean - p) <= step / 256 + 1e-12)
