"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong index, a swapped operand ...), builds that copy on the CPU and
runs the pin tests against it in a subprocess: every mutant must fail them.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "dropped_scale": ("scores[j] = scale * dot;", "scores[j] = dot;"),
    "causal_off_by_one": ("h / group, p + 1,", "h / group, p,"),
    "top_left_alignment": ("const int64_t p = (int64_t)lk - lq + i;", "const int64_t p = i;"),
    "gqa_modulo_mapping": ("h / group, p + 1,", "h % kv_heads, p + 1,"),
    "slot_without_block_size": ("block_table_row[pos / block_size] * block_size + pos % block_size",
                                "block_table_row[pos / block_size] + pos % block_size"),
    "unnormalised_weights": ("double w = exp(scores[j] - m) / denom;", "double w = exp(scores[j] - m);"),
    "reads_k_for_v": ("out[e] += w * vj[e];", "out[e] += w * kj[e];"),
    "decode_drops_new_token": ("&src, h / group, ctx,", "&src, h / group, ctx - 1,"),
    "bf16_widening_shift": ("((uint32_t)bits) << 16;", "((uint32_t)bits) << 15;"),
    "store_writes_k_to_v": ("v_cache[slot * row + e] = v[t * v_stride + e];",
                            "v_cache[slot * row + e] = k[t * k_stride + e];"),
    "store_drops_bounds_report": ("if (slot == -1) continue;", "if (slot < 0) continue;"),
    "rmsnorm_sum_not_mean": ("sqrt(ss / n + eps)", "sqrt(ss + eps)"),
    "rmsnorm_eps_outside_sqrt": ("sqrt(ss / n + eps)", "(sqrt(ss / n) + eps)"),
    "rope_adjacent_pairs": ("const double a = x[i], b = x[i + half];",
                            "const double a = x[(2 * i) % d], b = x[(2 * i + 1) % d];"),
    "rope_sin_sign": ("y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    "rope_frequency_exponent": ("pow(base, (2.0 * i) / d)", "pow(base, (1.0 * i) / d)"),
    "k_rotated_with_q_weight": ("d, k_weight, eps, cs, k_cache", "d, q_weight, eps, cs, k_cache"),
    "v_cache_gets_k": ("v_cache[slot * row + (int64_t)g * d + i] = tok[((int64_t)num_heads + kv_heads + g) * d + i];",
                       "v_cache[slot * row + (int64_t)g * d + i] = tok[((int64_t)num_heads + g) * d + i];"),
    "meta_start_ignores_cache": ("const int start = num_cached[b] < seqlen - 1 ? num_cached[b] : seqlen - 1;",
                                 "const int start = 0;"),
    "meta_keys_are_queries": ("const int seqlen_k = end;", "const int seqlen_k = seqlen_q;"),
    "meta_first_block_offset_dropped": ("if (i == start_block) slot_start += start % block_size;",
                                        "if (i == start_block) slot_start += 0;"),
    "meta_last_block_full": ("if (i == end_block - 1) slot_end = base + end - (int64_t)i * block_size;",
                             "if (i == end_block - 1) slot_end = base + block_size;"),
    "meta_decode_position_is_length": ("positions[b] = seqlen - 1;", "positions[b] = seqlen;"),
    "meta_decode_slot_first_block": ("block_table[(int64_t)b * max_blocks + last]", "block_table[(int64_t)b * max_blocks]"),
    "e4m3_exponent_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_subnormal_scale": ("ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)"),
    "e4m3_ties_away": ("int q = (int)nearbyint(ldexp(a, 3 - ex));", "int q = (int)round(ldexp(a, 3 - ex));"),
    "e4m3_no_saturation": ("if (a >= 448.0) return s | 0x7e;", "if (a >= 464.0) return s | 0x7f;"),
    "fp8_k_scale_dropped": ("kj[e] = e4m3_to_double(src->k8_cache[row + e]) * src->k_scale;",
                            "kj[e] = e4m3_to_double(src->k8_cache[row + e]);"),
    "fp8_store_multiplies": ("(uint8_t)orc_e4m3_encode(kx / k_scale);", "(uint8_t)orc_e4m3_encode(kx * k_scale);"),
    "rope_before_weight": ("x[i] = bf16_to_double(double_to_bf16(yn * bf16_to_double(w_bits[i])));",
                           "x[i] = yn;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new), encoding="utf-8")
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", str(mutant_c), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, PA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_norm_rope.py"),
                        os.path.join(ROOT, "tests", "test_oracle_metadata.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fp8.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
