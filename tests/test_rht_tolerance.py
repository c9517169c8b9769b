"""The RHT column-wise tolerance check itself (nvfp4_testutil.check_rht_columns),
on the CPU: the oracle's output passes with no difference; the output of the
same transform summed in another FP32 order (descending) passes, each
difference explained by a rounding tie; a code moved one E2M1 step where
no tie explains it, or a scale moved where no tie changes the block
maximum, fails; a code or a block scale moved where a tie does explain it
passes and is counted.  The tolerance follows the Hadamard quantize's
description ("Write both NVFP4 amax buffers", review reply on aliasing:
the column-wise amax is taken after the transform; codes may then differ
only where another summation order moves a rounding decision)."""
import numpy as np
import pytest
import torch

from nvfp4_testutil import check_rht_columns, rht_tie_candidates, unpack

MASK = 0x3C5A


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _pack(q: np.ndarray) -> np.ndarray:
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def _columns_as_kernel_would(oracle, xb, mask, t16_bits, amax_col):
    """Column-wise codes and compact scales of given transformed columns
    (BF16 bits, [N, M]) under the tensor's column amax: the 1D quantization
    of those rows, by the oracle."""
    a = float(amax_col)
    q = oracle.quantize("1d", t16_bits, colwise=False, amax=(a, a))
    return q["row_data"], q["row_scale"]


@pytest.fixture(scope="module")
def wide(oracle_mod):
    rng = np.random.default_rng(1)
    M, N = 512, 256
    xb = _bf16(rng.standard_normal((M, N)) * 2.0 ** rng.integers(-12, 8, (M, N)))
    return xb, oracle_mod.quantize("rht", xb, sign_mask=MASK)


def test_oracle_output_passes(oracle_mod, wide):
    xb, ref = wide
    c = check_rht_columns(oracle_mod, xb, MASK, ref["col_data"], ref["col_scale"], ref)
    assert c["codes_differing"] == 0 and c["scales_differing"] == 0
    assert c["tie_candidates"] > 0


def test_another_summation_order_passes(oracle_mod, wide):
    xb, ref = wide
    M, N = xb.shape
    X = (xb.astype(np.uint32) << 16).view(np.float32)
    H = oracle_mod.hadamard16().astype(np.float32)
    sign = np.array([-1.0 if (MASK >> i) & 1 else 1.0 for i in range(16)], np.float32)
    u = X.reshape(M // 16, 16, N) * sign[None, :, None]
    acc = np.zeros((M // 16, 16, N), np.float32)
    for i in range(15, -1, -1):                      # descending: not the oracle's order
        acc = acc + H[None, :, i, None] * u[:, i, None, :]
    t = _bf16((acc * np.float32(0.25)).reshape(M, N).T)
    assert np.any(t != _bf16(oracle_mod.rht_columns(xb, MASK, False)))   # some BF16 values do flip
    d, s = _columns_as_kernel_would(oracle_mod, xb, MASK, t, ref["amax_col"][0])
    check_rht_columns(oracle_mod, xb, MASK, d, s, ref)


def _integer_case(oracle_mod):
    # multiples of 1/8 below 16: every transform is exact in FP32, and many
    # are exact BF16 midpoints (ties)
    rng = np.random.default_rng(7)
    M, N = 256, 128
    xb = _bf16(rng.integers(-127, 128, (M, N)) / 8.0)
    return xb, oracle_mod.quantize("rht", xb, sign_mask=MASK)


def test_unexplained_code_fails(oracle_mod):
    xb, ref = _integer_case(oracle_mod)
    t16, alt, cand = rht_tie_candidates(oracle_mod, xb, MASK, np.arange(xb.shape[1]))
    q = unpack(ref["col_data"])
    k, y = np.argwhere(~cand & ((q & 7) > 0) & ((q & 7) < 7))[0]
    q[k, y] -= 1                                     # one E2M1 step toward zero, no tie there
    with pytest.raises(AssertionError, match="not explained"):
        check_rht_columns(oracle_mod, xb, MASK, _pack(q), ref["col_scale"], ref)


def test_code_flipped_at_a_tie_passes(oracle_mod):
    xb, ref = _integer_case(oracle_mod)
    N = xb.shape[1]
    t16, alt, cand = rht_tie_candidates(oracle_mod, xb, MASK, np.arange(N))
    g = oracle_mod.global_encode_scale(float(ref["amax_col"][0]))
    rtab = np.array([oracle_mod.encode_factor(s, g) for s in range(128)], np.float32)
    r = np.repeat(rtab[ref["col_scale"]], 16, axis=1)
    c_t = oracle_mod.encode_array(t16 * r, "e2m1")
    c_a = oracle_mod.encode_array(alt * r, "e2m1")
    # a tie whose other rounding changes the code but not its block's maximum
    bmax = np.repeat(np.abs(t16).reshape(N, -1, 16).max(-1), 16, axis=1)
    pick = np.argwhere(cand & (c_a != c_t) & (np.abs(alt) < bmax))
    assert pick.size > 0
    k, y = pick[0]
    q = unpack(ref["col_data"])
    q[k, y] = c_a[k, y]
    c = check_rht_columns(oracle_mod, xb, MASK, _pack(q), ref["col_scale"], ref)
    assert c["codes_differing"] == 1 and c["scales_differing"] == 0


def test_scale_moved_without_a_tie_fails(oracle_mod):
    xb, ref = _integer_case(oracle_mod)
    N = xb.shape[1]
    t16, alt, cand = rht_tie_candidates(oracle_mod, xb, MASK, np.arange(N))
    bcand = cand.reshape(N, -1, 16).any(-1)
    s = ref["col_scale"].copy()
    k, b = np.argwhere(~bcand & (s > 0) & (s < 0x7E))[0]
    s[k, b] += 1
    # the block's codes follow the moved scale, so only the scale is wrong
    g = oracle_mod.global_encode_scale(float(ref["amax_col"][0]))
    q = unpack(ref["col_data"])
    r = np.float32(oracle_mod.encode_factor(int(s[k, b]), g))
    q[k, 16 * b:16 * b + 16] = oracle_mod.encode_array(t16[k, 16 * b:16 * b + 16] * r, "e2m1")
    with pytest.raises(AssertionError, match="scale"):
        check_rht_columns(oracle_mod, xb, MASK, _pack(q), s, ref)


def test_block_maximum_at_a_tie_passes(oracle_mod):
    xb, ref = _integer_case(oracle_mod)
    N = xb.shape[1]
    t16, alt, cand = rht_tie_candidates(oracle_mod, xb, MASK, np.arange(N))
    g = oracle_mod.global_encode_scale(float(ref["amax_col"][0]))
    a = np.abs(t16).reshape(N, -1, 16)
    arg = a.argmax(-1)
    kk, bb = np.indices(arg.shape)
    at_max = cand.reshape(N, -1, 16)[kk, bb, arg]
    up = np.abs(alt).reshape(N, -1, 16)[kk, bb, arg] > a.max(-1)
    for k, b in np.argwhere(at_max & up):
        y = 16 * b + arg[k, b]
        s_new = oracle_mod.block_scale(float(abs(alt[k, y])), g)
        if s_new == ref["col_scale"][k, b]:
            continue
        # the kernel's block: the maximum rounded the other way, its scale and
        # every code of the block from that scale's encode factor
        t_blk = t16[k, 16 * b:16 * b + 16].copy()
        t_blk[arg[k, b]] = alt[k, y]
        r = np.float32(oracle_mod.encode_factor(s_new, g))
        q = unpack(ref["col_data"])
        q[k, 16 * b:16 * b + 16] = oracle_mod.encode_array(t_blk * r, "e2m1")
        s = ref["col_scale"].copy()
        s[k, b] = s_new
        c = check_rht_columns(oracle_mod, xb, MASK, _pack(q), s, ref)
        assert c["scales_differing"] == 1
        return
    pytest.fail("no block whose maximum sits at a tie that moves its scale")
