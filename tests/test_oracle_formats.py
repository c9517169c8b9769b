"""Pins of the oracle's number formats (E2M1, E4M3, BF16) and scale layouts
against facts that do not come from the oracle itself: the format
definitions (golden tables), independent library rounding routines (numpy's
round-half-even, PyTorch's FP8/BF16 casts) and exhaustive enumeration."""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------------------
# E2M1
# ---------------------------------------------------------------------------

def test_e2m1_golden_table(oracle_mod):
    for v, code in _read("e2m1_rounding.txt"):
        assert oracle_mod.e2m1(float(v)) == int(code), v


def test_e2m1_values(oracle_mod):
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = oracle_mod.e2m1_value(c)
        assert abs(v) == mags[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)
        # every code is a fixed point of encode(decode(.))
        assert oracle_mod.e2m1(v) == c


def _e2m1_by_rint(v: np.ndarray) -> np.ndarray:
    """Independent E2M1 encoder: numpy's round-half-even on the grid of each
    binade ([0,2): step 0.5, [2,4): step 1, [4,6): step 2), then saturation."""
    m = np.abs(v.astype(np.float64))
    val = np.where(m < 2.0, np.rint(m * 2.0) / 2.0,
                   np.where(m < 4.0, np.rint(m), np.where(m < 6.0, 2.0 * np.rint(m / 2.0), 6.0)))
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    code = np.vectorize(table.__getitem__)(val).astype(np.uint8)
    return code | np.where(np.signbit(v), 8, 0).astype(np.uint8)


def test_e2m1_exhaustive_bf16_vs_rint(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle_mod.encode_array(f, "e2m1")
    np.testing.assert_array_equal(got, _e2m1_by_rint(f))


def test_e2m1_boundaries_fp32_vs_rint(oracle_mod):
    # every decision point (midpoints and 6.0) and its FP32 neighbours
    pts = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1, 2, 4], dtype=np.float32)
    vals = []
    for p in pts:
        for k in range(-3, 4):
            q = p
            step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
            for _ in range(abs(k)):
                q = np.nextafter(q, step)
            vals += [q, -q]
    rng = np.random.default_rng(11)
    vals = np.concatenate([np.array(vals, dtype=np.float32),
                           rng.uniform(-8, 8, 20000).astype(np.float32)])
    np.testing.assert_array_equal(oracle_mod.encode_array(vals, "e2m1"), _e2m1_by_rint(vals))


# ---------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# E2M1 with stochastic rounding (one random byte per element)
# ---------------------------------------------------------------------------

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_sr_golden_table(oracle_mod):
    for line in _read("e2m1_sr.txt"):
        v, byte, code = float(line[0]), int(line[1]), int(line[2])
        assert oracle_mod.e2m1_sr(v, byte) == code, (v, byte)


def test_e2m1_sr_representable_values_never_move(oracle_mod):
    for c in range(16):
        v = oracle_mod.e2m1_value(c)
        got = oracle_mod.e2m1_sr_array(np.full(256, v, np.float32), np.arange(256, dtype=np.uint8))
        assert (got == c).all(), c


def test_e2m1_sr_up_count_is_ceil_256f(oracle_mod):
    """Over all 256 bytes, v between neighbours lo < v < hi rounds up for
    exactly ceil(256 f) of them, f = (v - lo) / (hi - lo) as an exact
    rational, and those are the smallest bytes (a threshold)."""
    from fractions import Fraction
    rb = np.arange(256, dtype=np.uint8)
    for lo, hi in zip(E2M1_GRID[:-1], E2M1_GRID[1:]):
        step = hi - lo
        cands = [lo + step * k / 256 for k in (1, 37, 128, 255)] + \
                [lo + step / 3, lo + step * 0.7071, np.nextafter(np.float32(lo), np.float32(7)),
                 np.nextafter(np.float32(hi), np.float32(0))]
        for v in np.array(cands, dtype=np.float32):
            f = (Fraction(float(v)) - Fraction(lo)) / Fraction(step)
            assert 0 < f < 1
            want_up = math.ceil(f * 256)
            got = oracle_mod.e2m1_sr_array(np.full(256, v, np.float32), rb)
            lo_code, hi_code = E2M1_GRID.index(lo), E2M1_GRID.index(hi)
            assert set(np.unique(got)) <= {lo_code, hi_code}
            up = got == hi_code
            assert int(up.sum()) == want_up, (float(v), lo, hi)
            assert up[:want_up].all()                       # the smallest bytes round up


def _e2m1_ceil(v: np.ndarray) -> np.ndarray:
    """Independent: the smallest E2M1 magnitude >= |v| (numpy searchsorted),
    saturated at 6, with the sign of v."""
    m = np.minimum(np.abs(v.astype(np.float64)), 6.0)
    code = np.searchsorted(np.array(E2M1_GRID), m, side="left").astype(np.uint8)
    return code | np.where(np.signbit(v), 8, 0).astype(np.uint8)


def test_e2m1_sr_zero_bytes_round_away_from_zero(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle_mod.e2m1_sr_array(f, np.zeros(f.size, np.uint8))
    np.testing.assert_array_equal(got, _e2m1_ceil(f))


def test_e2m1_sr_sign_and_saturation(oracle_mod):
    rng = np.random.default_rng(3)
    v = rng.uniform(0, 8, 4096).astype(np.float32)
    rb = rng.integers(0, 256, 4096).astype(np.uint8)
    pos = oracle_mod.e2m1_sr_array(v, rb)
    neg = oracle_mod.e2m1_sr_array(-v, rb)
    np.testing.assert_array_equal(neg, pos | 8)
    assert (pos[v >= 6] == 7).all()
    assert oracle_mod.e2m1_sr(-0.0, 0) == 8 and oracle_mod.e2m1_sr(float("inf"), 0) == 7


def test_e4m3_golden_table(oracle_mod):
    for kind, a, b in _read("e4m3_values.txt"):
        if kind == "decode":
            assert oracle_mod.e4m3_value(int(a, 16)) == float(b), a
        else:
            assert oracle_mod.e4m3(float(a)) == int(b, 16), a


def test_e4m3_decode_matches_torch(oracle_mod):
    codes = torch.arange(0, 127, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(int(c)) for c in codes])
    np.testing.assert_array_equal(got, ref)


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_exhaustive_bf16_vs_torch(oracle_mod):
    # every non-negative BF16 value up to 448 (PyTorch's cast does not
    # saturate, so the comparison stops at the largest finite value)
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    f = f[f <= 448.0]
    np.testing.assert_array_equal(oracle_mod.encode_array(f, "e4m3"), _torch_e4m3(f))


def test_e4m3_encode_midpoints_vs_torch(oracle_mod):
    vals = [oracle_mod.e4m3_value(c) for c in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    pts = []
    for m in mids + vals:
        q = np.float32(m)
        pts += [q, np.nextafter(q, np.float32(np.inf)), np.nextafter(q, np.float32(0))]
    rng = np.random.default_rng(5)
    pts = np.concatenate([np.array(pts, dtype=np.float32),
                          np.exp(rng.uniform(np.log(1e-4), np.log(448), 50000)).astype(np.float32)])
    pts = pts[pts <= 448.0]
    np.testing.assert_array_equal(oracle_mod.encode_array(pts, "e4m3"), _torch_e4m3(pts))


def test_e4m3_saturates(oracle_mod):
    for v in [448.00003, 450.0, 479.9, 480.0, 1e6, 3.0e38, float("inf")]:
        assert oracle_mod.e4m3(v) == 0x7E


# ---------------------------------------------------------------------------
# BF16
# ---------------------------------------------------------------------------

def test_bf16_round_matches_torch(oracle_mod):
    rng = np.random.default_rng(3)
    base = rng.standard_normal(20000).astype(np.float32) * np.float32(37.0)
    # exact ties: a BF16 value plus half a BF16 ulp, odd and even lsb
    b = (rng.integers(0x3000, 0x4F00, 2000).astype(np.uint32) << 16)
    ties = (b | 0x8000).view(np.float32)
    near = np.concatenate([(b | 0x7FFF).view(np.float32), (b | 0x8001).view(np.float32)])
    vals = np.concatenate([base, ties, -ties, near, np.array([0.0, -0.0, 3.0e38, -3.0e38], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle_mod.encode_array(vals, "bf16"), ref)


# ---------------------------------------------------------------------------
# Scale layout
# ---------------------------------------------------------------------------

def test_swizzle_golden_offsets(oracle_mod):
    for R, C, r, c, off in _read("swizzle_offsets.txt"):
        assert oracle_mod.swizzle_offset(int(r), int(c), int(C)) == int(off)


def _swizzle_by_reshape(compact: np.ndarray) -> np.ndarray:
    """The layout built from its description alone: cut into 128x4 tiles in
    row-major tile order; a tile's rows j*32 + i (j = 0..3) form line i."""
    R, C = compact.shape
    t = compact.reshape(R // 128, 128, C // 4, 4).transpose(0, 2, 1, 3)   # tiles [tr][tc][128][4]
    t = t.reshape(R // 128, C // 4, 4, 32, 4).transpose(0, 1, 3, 2, 4)      # [tr][tc][i][j][c]
    return np.ascontiguousarray(t).reshape(-1)


@pytest.mark.parametrize("R,C", [(128, 4), (256, 8), (384, 12), (128, 64)])
def test_swizzle_is_the_tiled_permutation(oracle_mod, R, C):
    rng = np.random.default_rng(R * 7 + C)
    compact = rng.integers(0, 256, (R, C), dtype=np.uint8)
    np.testing.assert_array_equal(oracle_mod.swizzle(compact), _swizzle_by_reshape(compact))
    # a bijection on [0, R*C)
    offs = sorted(oracle_mod.swizzle_offset(r, c, C) for r in range(R) for c in range(C))
    assert offs == list(range(R * C))
    # the four scales of one row inside a tile are contiguous (one 32-bit store)
    for r in range(0, R, 37):
        for c0 in range(0, C, 4):
            o = [oracle_mod.swizzle_offset(r, c0 + k, C) for k in range(4)]
            assert o == list(range(o[0], o[0] + 4)) and o[0] % 4 == 0


def test_swizzle_rejects_unaligned(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.swizzle(np.zeros((120, 4), np.uint8))
    with pytest.raises(ValueError):
        oracle_mod.swizzle(np.zeros((128, 6), np.uint8))


# ---------------------------------------------------------------------------
# Hadamard
# ---------------------------------------------------------------------------

def test_hadamard_is_sylvester(oracle_mod):
    H = oracle_mod.hadamard16()
    H2 = np.array([[1, 1], [1, -1]])
    ref = np.kron(np.kron(np.kron(H2, H2), H2), H2)
    np.testing.assert_array_equal(H, ref)
    np.testing.assert_array_equal(H @ H.T, 16 * np.eye(16, dtype=np.int64))


def test_rht16_small_integers_exact(oracle_mod):
    H = oracle_mod.hadamard16().astype(np.float64)
    rng = np.random.default_rng(9)
    for trial in range(200):
        v = rng.integers(-64, 65, 16).astype(np.float32)
        mask = int(rng.integers(0, 1 << 16))
        sign = np.array([-1.0 if (mask >> i) & 1 else 1.0 for i in range(16)])
        ref = H @ (sign * v) / 4.0   # exact: integer sums, then a power-of-two divide
        np.testing.assert_array_equal(oracle_mod.rht16(v, mask, round_bf16=False), ref.astype(np.float32))


def test_rht16_unit_and_constant_vectors(oracle_mod):
    for i in range(16):
        e = np.zeros(16, np.float32)
        e[i] = 1.0
        t = oracle_mod.rht16(e, 0, False)
        assert np.all(np.abs(t) == 0.25)
    t = oracle_mod.rht16(np.full(16, 3.0, np.float32), 0, False)
    assert t[0] == 12.0 and np.all(t[1:] == 0.0)
    # the transform is orthonormal after the 1/4: applying it twice returns v
    v = np.arange(16, dtype=np.float32) - 7.0
    np.testing.assert_array_equal(oracle_mod.rht16(oracle_mod.rht16(v, 0, False), 0, False), v)


def test_rht16_bf16_rounding(oracle_mod):
    rng = np.random.default_rng(4)
    for _ in range(100):
        v = torch.randn(16).to(torch.bfloat16).float().numpy()
        t32 = oracle_mod.rht16(v, 0xA5A5, False)
        t16 = oracle_mod.rht16(v, 0xA5A5, True)
        ref = torch.from_numpy(t32).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(t16, ref)


def test_printed_rht_amaxes_are_bf16_numbers(oracle_mod):
    # the reading "t is rounded to BF16 before the amax" rests on this
    for name, row, col in _read("rht_printed_amax.txt"):
        for v in (float(row), float(col)):
            assert float(torch.tensor(v).to(torch.bfloat16)) == v
