"""Plants plausible mistakes in copies of the oracle (on the CPU) and checks
that each one fails at least one pin of ``test_oracle_pins``.  A mutation
whose target text is missing fails the test, so the list stays in step with
``oracle/oracle.c``."""

import os

import pytest

import oracle
from tests.test_oracle_pins import PINS

MUTANTS = {
    "gqa_head_map_modulo": ("attend(qt, kc, vc, n, h / group,", "attend(qt, kc, vc, n, h % num_kv_heads,"),
    "page_offset_dropped": ("(int64_t)page * block_size + j % block_size", "(int64_t)page * block_size"),
    "logical_not_physical_page": ("int64_t r = (int64_t)page * block_size", "int64_t r = (int64_t)logical * block_size"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "no_normalisation": ("out[d] /= l;", "out[d] /= 1.0f;"),
    "exp_sign_flipped": ("s[j] = expf(s[j] - m);", "s[j] = expf(m - s[j]);"),
    "v_gathered_from_k": ("vc[j * row + e] = to_float(v_cache[r * row + e], dtype);",
                          "vc[j * row + e] = to_float(k_cache[r * row + e], dtype);"),
    "causal_top_left": ("attend(qt, kc, vc, prefix + r + 1,", "attend(qt, kc, vc, r + 1,"),
    "causal_off_by_one": ("attend(qt, kc, vc, prefix + r + 1,", "attend(qt, kc, vc, prefix + r + (r > 0),"),
    "chunk_rows_ignore_seq_offset": ("to_float(k[(q0 + r) * row + e], dtype)", "to_float(k[(r) * row + e], dtype)"),
    "store_v_from_k": ("v_cache[s * row + e] = v[t * v_row_stride + e];", "v_cache[s * row + e] = k[t * k_row_stride + e];"),
    "store_ignores_row_stride": ("k_cache[s * row + e] = k[t * k_row_stride + e];", "k_cache[s * row + e] = k[t * row + e];"),
    "bf16_shift_wrong": ("(uint32_t)h << 16;", "(uint32_t)h << 15;"),
    "f16_bias_wrong": ("e - 25);", "e - 24);"),
    "f16_subnormal_wrong": ("ldexpf((float)m, -24);", "ldexpf((float)m, -25);"),
    "sample_noise_multiplies": ("const float score = p / (e > 1e-10f ? e : 1e-10f);",
                                "const float score = p * (e > 1e-10f ? e : 1e-10f);"),
    "sample_temperature_ignored": ("const float a = x / t;\n            if (!(a > -INFINITY))\n                continue;",
                                   "const float a = x;\n            if (!(a > -INFINITY))\n                continue;"),
    "sample_last_index_on_ties": ("if (score > best) {", "if (score >= best) {"),
    "e4m3_bias_wrong": ("v = ldexpf((float)(m + 8), e - 10);", "v = ldexpf((float)(m + 8), e - 9);"),
    "e4m3_subnormal_wrong": ("v = ldexpf((float)m, -9);", "v = ldexpf((float)m, -10);"),
    "e4m3_ties_to_odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    "fp8_store_multiplies_scale": ("float_to_e4m3(to_float(k[t * k_row_stride + e], dtype) / k_scale)",
                                   "float_to_e4m3(to_float(k[t * k_row_stride + e], dtype) * k_scale)"),
    "fp8_decode_drops_v_scale": ("vc[j * row + e] = e4m3_to_float(v_cache[r * row + e]) * v_scale;",
                                 "vc[j * row + e] = e4m3_to_float(v_cache[r * row + e]);"),
    "minus_one_block_read_as_block_0": ("if (page < 0 || page >= num_blocks)\n        return -1;",
                                        "if (page >= num_blocks)\n        return -1;\n    if (page < 0) page = 0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SRC) as f:
        src = f.read()
    assert old in src, f"mutation target for {name} not found in oracle.c"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.load(oracle.build(str(mutated), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (KeyboardInterrupt, SystemExit):
            raise
        except BaseException:  # an assertion, an oracle error or pytest.raises' failure all count
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
