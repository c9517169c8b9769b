"""The test harness's own pieces, on the CPU: the slab-parallel oracle
(oracle_quantize_slabs) returns exactly what one whole-tensor oracle call
returns, for every mode and both directions; the scale read-back from the
128x4 layout inverts the oracle's permutation."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_amax_gb300 import inputs
from nvfp4_testutil import bits, oracle_quantize_slabs, scales_compact


@pytest.mark.parametrize("mode", ["1d", "2d", "rht", "row_scaled"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_slabs_equal_one_call(oracle_mod, mode, dtype):
    if mode == "rht" and dtype == torch.float32:
        pytest.skip("RHT takes BF16")
    M, N = 400, 272
    kind = inputs.row_mix if mode == "row_scaled" else inputs.outliers
    xb = bits(kind(M, N, seed=3, frac=0.05, dtype=dtype))
    colwise = mode != "row_scaled"
    mask = 0xA55A if mode == "rht" else 0
    whole = oracle_mod.quantize(mode, xb, colwise=colwise, sign_mask=mask)
    slabs = oracle_quantize_slabs(oracle_mod, mode, xb, colwise=colwise, sign_mask=mask, workers=5)
    keys = ["row_data", "row_scale", "amax_row"] + (["col_data", "col_scale", "amax_col"] if colwise else [])
    for k in keys:
        np.testing.assert_array_equal(slabs[k], whole[k], err_msg=k)


def test_scales_compact_inverts_the_swizzle(oracle_mod):
    rng = np.random.default_rng(0)
    for R, C in [(128, 4), (256, 40), (1024, 8)]:
        c = rng.integers(0, 256, (R, C), dtype=np.uint8)
        np.testing.assert_array_equal(scales_compact(oracle_mod, oracle_mod.swizzle(c), R, C, True), c)
        np.testing.assert_array_equal(scales_compact(oracle_mod, c.reshape(-1), R, C, False), c)
