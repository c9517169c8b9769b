"""Planted mistakes: each must make one of the oracle's pins fail.

Each case below alters one step of ``oracle/nvfp4_oracle.c`` the way a
plausible slip would (a wrong constant, a dropped term, a swapped index, the
wrong tie rule), compiles the altered copy with gcc and runs the pin files
(``test_oracle_formats.py``, ``test_oracle_quantize.py``) against it in a
child process.  The pins are only worth trusting if every such copy fails
them.  An unaltered copy built the same way must pass, so a failure here
cannot come from the mechanism itself.  Everything runs on the CPU.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_formats.py"),
        os.path.join(ROOT, "tests", "test_oracle_quantize.py")]

# name -> (original text, altered text); each original occurs exactly once.
MUTANTS = {
    # global encode scale 448*6/amax: dropped the E2M1 maximum
    "global_scale_without_6": ("float g = 2688.0f / amax;", "float g = 448.0f / amax;"),
    # amax = 0 reading: g = 1
    "zero_amax_scale": ("if (amax == 0.0f) return 1.0f;", "if (amax == 0.0f) return 0.0f;"),
    # block scale b/6*g: wrong E2M1 maximum
    "block_scale_over_4": ("float q = block_amax / 6.0f;", "float q = block_amax / 4.0f;"),
    # block scale order of the FP32 operations: (b*g)/6 instead of (b/6)*g
    "block_scale_order": ("float q = block_amax / 6.0f;\n  float sf = q * g;",
                          "float q = block_amax * g;\n  float sf = q / 6.0f;"),
    # encode factor g/s inverted
    "encode_factor_inverted": ("float r = g / sv;", "float r = sv / g;"),
    # blocks whose scale is 0 must encode to 0, not saturate
    "zero_scale_block": ("if (s == 0) return 0.0f;", "if (s == 0) return FLT_MAX;"),
    # E2M1 ties: away from zero instead of to even
    "e2m1_ties_away": ("(d == best_d && (c & 1) == 0)) {\n      best = c;\n      best_d = d;\n    }\n  }\n"
                       "  return (uint8_t)(sign | (uint8_t)best);",
                       "(d == best_d)) {\n      best = c;\n      best_d = d;\n    }\n  }\n"
                       "  return (uint8_t)(sign | (uint8_t)best);"),
    # E4M3 saturation bound
    "e4m3_no_saturation": ("if (x > 448.0) return 0x7E;", "if (x > 448.0) return 0x7F;"),
    # E4M3 exponent bias 8 instead of 7
    "e4m3_bias": ("v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    # BF16 rounding: ties up instead of to even
    "bf16_ties_up": ("if (rem > 0x8000u || (rem == 0x8000u && (hi & 1u))) hi += 1u;",
                     "if (rem >= 0x8000u) hi += 1u;"),
    # element 2i in the high nibble instead of the low one
    "nibble_order": ("if (j & 1)\n    row[j >> 1]", "if (!(j & 1))\n    row[j >> 1]"),
    # dequantize reads nibbles the other way round
    "dequant_nibble_order": ("uint8_t q = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);",
                             "uint8_t q = (j & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);"),
    # dequantize by a/448 instead of a/(448*6)
    "dequant_scale": ("float k = a / 2688.0f;", "float k = a / 448.0f;"),
    # 2D: tile maximum over one row of the tile only
    "tile_max_one_row": ("for (int dy = 0; dy < 16; ++dy)\n      for (int i = 0; i < 16; ++i) {",
                         "for (int dy = 0; dy < 1; ++dy)\n      for (int i = 0; i < 16; ++i) {"),
    # RHT: column-wise codes scaled by the row-wise (untransformed) amax
    "rht_column_global_scale": ("quantize_vector_1d(vec, M, g_col, rbits", "quantize_vector_1d(vec, M, g_row, rbits"),
    # row-scaled: the tensor's amax instead of the row's
    "row_scaled_tensor_amax": ("float g = oracle_global_encode_scale(a);",
                               "float g = oracle_global_encode_scale(oracle_amax(x, dtype, M * N));"),
    # column gather transposed the wrong way
    "column_index": ("col[y] = load_elem(x, dtype, y * N + j);", "col[y] = load_elem(x, dtype, j * M + y);"),
    # RHT: (1/2) instead of (1/4)
    "rht_normalisation": ("float r = acc * 0.25f;", "float r = acc * 0.5f;"),
    # RHT: not a Hadamard matrix (popcount of o|i)
    "hadamard_entry": ("for (int b = o & i; b; b >>= 1)", "for (int b = o | i; b; b >>= 1)"),
    # RHT: sign bits read in reverse order
    "rht_sign_bit_order": ("u[i] = ((mask >> i) & 1u) ? -v[i] : v[i];",
                           "u[i] = ((mask >> (15 - i)) & 1u) ? -v[i] : v[i];"),
    # RHT: column amax taken before the transform
    "rht_amax_untransformed": ("amax_col = (mode == MODE_RHT) ? oracle_rht_amax(x, dtype, M, N, sign_mask) : amax_row;",
                               "amax_col = amax_row;"),
    # RHT columns exposed for the tolerance check: a block read one row off
    "rht_columns_row_offset": ("for (int i = 0; i < 16; ++i) v[i] = load_elem(x, dtype, (16 * b + i) * N + j);\n"
                               "      rht_block(v, mask, round_bf16",
                               "for (int i = 0; i < 16; ++i) v[i] = load_elem(x, dtype, (16 * b + (i + 1) % 16) * N + j);\n"
                               "      rht_block(v, mask, round_bf16"),
    # swizzle: the two row terms of the 128x4 tile swapped
    "swizzle_row_terms": ("(r % 32) * 16 + ((r % 128) / 32) * 4", "(r % 32) * 4 + ((r % 128) / 32) * 16"),
    # stochastic rounding: a byte equal to 256 f also rounds up
    "sr_threshold_inclusive": ("int up = (double)rb < f * 256.0;", "int up = (double)rb <= f * 256.0;"),
    # stochastic rounding: the sign of x dropped
    "sr_sign_dropped": ("return (uint8_t)(sign | (uint8_t)(lo + up));", "return (uint8_t)(lo + up);"),
    # stochastic rounding: the fraction measured in steps of 0.5 in every binade
    "sr_fixed_step": ("double f = (m - E2M1_MAG[lo]) / (E2M1_MAG[lo + 1] - E2M1_MAG[lo]);",
                      "double f = (m - E2M1_MAG[lo]) / 0.5;"),
    # stochastic rounding: the column-wise output reads the bytes of x^T's layout
    "sr_column_byte_index": ("quantize_vector_1d(vec, M, g_col, rbits ? rbits + j : NULL, N,",
                             "quantize_vector_1d(vec, M, g_col, rbits ? rbits + j * M : NULL, 1,"),
}


def _build(path, text):
    src = path + ".c"
    with open(src, "w") as f:
        f.write(text)
    import oracle
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", path, src, "-lm"])
    return path


def _run_pins(lib):
    env = dict(os.environ, NVFP4_ORACLE_LIB=lib)
    p = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return p.returncode, (p.stdout + p.stderr)[-600:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    d = tmp_path_factory.mktemp("oracle_mutants")
    with open(SRC) as f:
        text = f.read()
    jobs = {"unaltered": text}
    for name, (old, new) in MUTANTS.items():
        assert text.count(old) == 1, name
        jobs[name] = text.replace(old, new)
    libs = {name: _build(str(d / f"liboracle_{name}.so"), t) for name, t in jobs.items()}
    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {name: ex.submit(_run_pins, lib) for name, lib in libs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unaltered_copy_passes_the_pins(outcomes):
    rc, tail = outcomes["unaltered"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, tail = outcomes[name]
    assert rc == 1, f"{name}: pins passed or errored (rc={rc})\n{tail}"


# Planted mistakes in the grouped (multi-tensor) composition, which is Python:
# each altered version of ``quantize_grouped`` must fail one of the grouped
# pins of ``test_oracle_quantize.py``.
def _grouped_mutants(oracle):
    def shared_amax(mode, x, splits, rowwise=True, colwise=True):
        a = oracle.amax(x)
        out, r = [], 0
        for m in splits:
            out.append(oracle.quantize(mode, x[r:r + m], rowwise=rowwise, colwise=colwise, amax=(a, a)))
            r += m
        return out

    def rows_from_zero(mode, x, splits, rowwise=True, colwise=True):
        return [oracle.quantize(mode, x[:m], rowwise=rowwise, colwise=colwise) for m in splits]

    def columns_of_whole_tensor(mode, x, splits, rowwise=True, colwise=True):
        whole = oracle.quantize(mode, x, rowwise=False, colwise=colwise)
        out, r = [], 0
        for m in splits:
            o = oracle.quantize(mode, x[r:r + m], rowwise=rowwise, colwise=colwise)
            if colwise and m:
                o["col_data"] = whole["col_data"][:, r // 2:(r + m) // 2]
                o["col_scale"] = whole["col_scale"][:, r // 16:(r + m) // 16]
            out.append(o)
            r += m
        return out

    return {"shared_amax": shared_amax, "rows_from_zero": rows_from_zero,
            "columns_of_whole_tensor": columns_of_whole_tensor}


@pytest.mark.parametrize("name", ["shared_amax", "rows_from_zero", "columns_of_whole_tensor"])
def test_planted_grouped_mistake_fails_a_pin(name):
    import types

    import oracle
    import test_oracle_quantize as pins

    fake = types.SimpleNamespace(**{k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("__")})
    fake.quantize_grouped = _grouped_mutants(oracle)[name]
    checks = [pins.test_grouped_members_match_restatement, pins.test_grouped_2d_member_matches_restatement,
              pins.test_grouped_single_member_is_the_plain_quantize, pins.test_grouped_members_are_independent]
    failed = 0
    for check in checks:
        try:
            check(fake)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed > 0, f"no grouped pin caught {name}"
