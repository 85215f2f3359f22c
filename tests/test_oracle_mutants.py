"""Plant plausible mistakes in copies of the oracle source (on the CPU, in a
temporary directory) and check that at least one pin catches each of them.
The oracle itself is not modified."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tf_oracle.c")

MUTANTS = {
    "scatter_row_uses_head_group": ("(int64_t)r * Sl + t) * Hl + h) * D + d", "(int64_t)g * Sl + t) * Hl + h) * D + d"),
    "scatter_strided_head_band": ("(int64_t)(g * Hl + h) * sh + d;", "(int64_t)(h * P + g) * sh + d;"),
    "gather_strided_head_band": ("* H + g * Hl + h) * D + d;", "* H + h * P + g) * D + d;"),
    "gather_token_block_of_group": ("((int64_t)r * Sl + t) * at", "((int64_t)g * Sl + t) * at"),
    "rmsnorm_drops_eps": ("sqrtf(ms + eps)", "sqrtf(ms)"),
    "rmsnorm_sum_not_mean": ("(float)(ss / D)", "(float)(ss)"),
    "rmsnorm_squares_in_fp32": ("ss += (double)xf[d] * (double)xf[d];", "ss += (double)(xf[d] * xf[d]);"),
    "rmsnorm_mean_clamped_to_fp32": ("float ms = (float)(ss / D);", "float ms = (float)fmin(ss / D, FLT_MAX);"),
    "rmsnorm_no_cast_before_scale": ("y[d] = round16(fmt, prod);", "y[d] = prod;"),
    "rmsnorm_weight_dropped": ("y[d] * (float)tfo_decode16(fmt, w[d])", "y[d] * 1.0f"),
    "rope_wrong_sign": ("(double)(ac - bs)", "(double)(ac + bs)"),
    "rope_cos_sin_swapped": ("float c = cs[2 * i], s = cs[2 * i + 1];", "float s = cs[2 * i], c = cs[2 * i + 1];"),
    "rope_half_split_pairs": ("float a = z[2 * i], b = z[2 * i + 1];", "float a = z[i], b = z[i + D / 2];"),
    "rope_wrong_frequency": ("pow(theta, -2.0 * i / D)", "pow(theta, -1.0 * i / D)"),
    "rope_local_position": ("int64_t p = (int64_t)r * Sl + t;", "int64_t p = t;"),
    "codec_truncates": ("nearbyint(", "floor("),
    "neox_partner_adjacent": ("float first = z[i], second = z[i + half];", "float first = z[i], second = z[i + 1];"),
    "neox_wrong_sign": ("(double)(fc - ss_)", "(double)(fc + ss_)"),
    "neox_table_entry_of_element": ("float cos_i = cs[2 * i], sin_i = cs[2 * i + 1];",
                                    "float cos_i = cs[i], sin_i = cs[i + 1];"),
    "neox_style_ignored_in_scatter": ("        if (neox)\n", "        if (0)\n"),
    "projection_transposed_weight": ("const uint16_t *wn = w + (int64_t)n * w_row;", "const uint16_t *wn = w + n;"),
    "projection_drops_last_term": ("for (int k = 0; k < K; ++k)\n            acc +=", "for (int k = 0; k < K - 1; ++k)\n            acc +="),
    "projection_truncates": ("out[n - n0] = tfo_encode16(fmt, acc);", "out[n - n0] = tfo_encode16(fmt, (float)(int)acc);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    with open(SRC) as f:
        text = f.read()
    old, new = MUTANTS[name]
    assert text.count(old) == 1, f"mutation site for {name} not unique/found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so"), force=True))
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            caught.append(check.__name__)
            break
    assert caught, f"no pin caught the planted mistake {name}"
