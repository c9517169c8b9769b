"""The kernels' number-format building blocks on the GPU, compared with the
oracle exhaustively: hardware E2M1 / E4M3 / BF16 conversions, the
stochastic-rounding E2M1 encoder, the FMA-
corrected division by 6 against IEEE division over every positive FP32
value, and the bounded mbarrier wait giving up on a barrier nobody signals."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_testutil import build_selftest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def st():
    return build_selftest()


def _run(fn, vals: np.ndarray, out_dtype):
    x = torch.from_numpy(np.ascontiguousarray(vals, np.float32)).cuda()
    out = torch.empty(x.numel(), dtype=out_dtype, device="cuda")
    assert fn(x.data_ptr(), out.data_ptr(), x.numel()) == 0
    return out.cpu().numpy()


def _neighbourhoods(points, width):
    f = np.asarray(points, np.float32).view(np.uint32).astype(np.int64)
    idx = (f[:, None] + np.arange(-width, width + 1)[None, :]).ravel()
    idx = idx[(idx >= 0) & (idx < 0x7F800000)].astype(np.uint32)
    v = idx.view(np.float32)
    return np.concatenate([v, -v])


def _pad8(v):
    return np.concatenate([v, np.zeros((-v.size) % 8, np.float32)])


def test_e2m1_cvt_matches_oracle(st, oracle_mod):
    bf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1.0, 2.0, 4.0]
    rng = np.random.default_rng(0)
    vals = _pad8(np.concatenate([bf, _neighbourhoods(mids, 4096), rng.uniform(-7, 7, 1 << 20).astype(np.float32),
                                 np.array([0.0, -0.0, 1e-30, -1e-30, 3e38, -3e38, np.inf, -np.inf], np.float32)]))
    got = _run(st.selftest_e2m1, vals, torch.uint8)
    ref = oracle_mod.encode_array(vals, "e2m1")
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. {vals[bad[:5]]} -> gpu {got[bad[:5]]} oracle {ref[bad[:5]]}"


def test_e2m1_sr_encoder_matches_oracle(st, oracle_mod):
    """The stochastic-rounding encoder (carry form) against the oracle's
    rule: every finite BF16 value with every byte, the neighbourhoods of the
    points lo + b/256 (hi - lo) of every interval and byte (where a fraction
    just above b/256 must still round up: values whose low bits the carry
    form's truncation drops), and random FP32 values with random bytes."""
    bf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    pts = np.array([lo + (hi - lo) * b / 256 for lo, hi in zip(mags[:-1], mags[1:]) for b in range(256)])
    near = _neighbourhoods(pts[pts > 0], 3)
    rng = np.random.default_rng(3)
    rnd = (rng.choice([-1.0, 1.0], 1 << 22) * np.exp2(rng.uniform(-30, 4, 1 << 22))).astype(np.float32)
    special = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-38, 6.0, -6.0, 7.9, 3e38, -3e38, np.inf, -np.inf], np.float32)
    cases = [(np.repeat(bf, 256), np.tile(np.arange(256, dtype=np.uint8), bf.size)),
             (np.repeat(near, 256), np.tile(np.arange(256, dtype=np.uint8), near.size)),
             (rnd, rng.integers(0, 256, rnd.size).astype(np.uint8)),
             (np.repeat(special, 256), np.tile(np.arange(256, dtype=np.uint8), special.size))]
    for vals, rb in cases:
        x = torch.from_numpy(np.ascontiguousarray(vals, np.float32)).cuda()
        r = torch.from_numpy(np.ascontiguousarray(rb, np.uint8)).cuda()
        out = torch.empty(x.numel(), dtype=torch.uint8, device="cuda")
        assert st.selftest_e2m1_sr(x.data_ptr(), r.data_ptr(), out.data_ptr(), x.numel()) == 0
        got = out.cpu().numpy()
        ref = oracle_mod.e2m1_sr_array(vals, rb)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (f"{bad.size} of {vals.size} differ, e.g. {vals[bad[:5]]} bytes {rb[bad[:5]]} -> "
                               f"gpu {got[bad[:5]]} oracle {ref[bad[:5]]}")


def test_e4m3_cvt_matches_oracle(st, oracle_mod):
    bf = (np.arange(0x7F80, dtype=np.uint32) << 16).view(np.float32)
    vals = [oracle_mod.e4m3_value(c) for c in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    pts = _neighbourhoods(mids + vals + [448.0, 464.0, 480.0], 256)
    pts = pts[~np.signbit(pts)]   # block scales come from max|x| >= +0
    rng = np.random.default_rng(1)
    allv = np.concatenate([bf, pts, np.exp(rng.uniform(np.log(1e-6), np.log(1e4), 1 << 20)).astype(np.float32),
                           np.array([np.inf, 3e38], np.float32)])
    got = _run(st.selftest_e4m3, allv, torch.uint8)
    ref = oracle_mod.encode_array(allv, "e4m3")
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. {allv[bad[:5]]}"


def test_bf16_round_matches_oracle(st, oracle_mod):
    rng = np.random.default_rng(2)
    b = rng.integers(0, 0x7F7F, 1 << 18).astype(np.uint32) << 16
    vals = np.concatenate([(b | rng.integers(0, 0x10000, b.size).astype(np.uint32)).view(np.float32),
                           (b | 0x8000).view(np.float32)])
    vals = np.concatenate([vals, -vals])
    got = _run(st.selftest_bf16, vals, torch.int16).view(np.uint16)
    np.testing.assert_array_equal(got, oracle_mod.encode_array(vals, "bf16"))


def test_div6_is_ieee_division_for_every_positive_float(st):
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    ex = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert st.selftest_div6(0, 0x7F800000, bad.data_ptr(), ex.data_ptr()) == 0
    assert int(bad.item()) == 0, f"first mismatch at bits {int(ex.item()) & 0xFFFFFFFF:#x}"


def test_bounded_wait_gives_up_and_reports(st):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    result = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    # about 10 ms at the boost clock
    assert st.selftest_wait_timeout(status.data_ptr(), 20_000_000, result.data_ptr()) == 0
    assert int(result.item()) == 0
    assert int(status.item()) == 1
    # the context is still usable
    assert torch.ones(4, device="cuda").sum().item() == 4.0
