"""The pins must catch a plausible slip in the oracle. Each case copies
oracle.c, plants one mistake by text substitution, builds the copy with gcc
and runs the pin suite against it in a child process: the suite has to fail.
CPU only; nothing here touches the real oracle build."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rope_sign": ("out[i] = y[i] * c - y[i + half] * s;", "out[i] = y[i] * c + y[i + half] * s;"),
    "rope_pairing": ("out[i + half] = y[i + half] * c + y[i] * s;",
                     "out[i + half] = y[i + half] * c + y[i + 1] * s;"),
    "rope_frequency": ("-2.0 * (double)i / (double)rotary_dim", "-1.0 * (double)i / (double)rotary_dim"),
    "eps_outside_root": ("sqrt(sum_sq / head_dim + eps)", "(sqrt(sum_sq / head_dim) + eps)"),
    "norm_weight_dropped": ("y[d] = x[d] * inv_rms * w[d];", "y[d] = x[d] * inv_rms;"),
    "gqa_mapping": ("uint32_t kv_head = h / group;", "uint32_t kv_head = h % num_kv_heads;"),
    "window_off_by_one": ("start = L - sliding_window;", "start = L - sliding_window + 1;"),
    "k_scale_dropped": ("return oracle_e4m3_to_f64(k_cache_fp8[idx]) * (double)k_scale;",
                        "return oracle_e4m3_to_f64(k_cache_fp8[idx]);"),
    "e4m3_exponent_bias": ("v = ldexp(1.0 + m / 8.0, ef - 7);", "v = ldexp(1.0 + m / 8.0, ef - 8);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_ties_away": ("double y = rint(ax / quantum) * quantum; /* at most 448",
                       "double y = round(ax / quantum) * quantum; /* at most 448"),
    "e4m3_no_saturation": ("if (ax >= 448.0) return (uint8_t)(sign | 0x7Eu);",
                           "if (ax >= 464.0) return 0x7Fu;"),
    "bf16_double_rounding": ("double n = rint(ax / quantum);",
                             "double n = rint((double)(float)ax / quantum);"),
    "bf16_rows_at_packed_stride": ("value[(int64_t)t * value_stride + (int64_t)h * head_dim + d];",
                                   "value[(int64_t)t * num_kv_heads * head_dim + (int64_t)h * head_dim + d];"),
    "slot_row": ("slots[i] = physical_block * (int64_t)block_size + (int64_t)(p % block_size);",
                 "slots[i] = physical_block * (int64_t)block_size + (int64_t)(i % block_size);"),
    "pool_head_major": ("return ((block * (int64_t)block_size + offset) * num_kv_heads + head) * (int64_t)head_dim + d;",
                        "return ((block * (int64_t)num_kv_heads + head) * block_size + offset) * (int64_t)head_dim + d;"),
    "value_row_of_key": ("acc[d] += e * value_at(v_cache, v_cache_fp8,",
                         "acc[d] += e * value_at(k_cache_bf16 ? k_cache_bf16 : v_cache, v_cache_fp8,"),
    "v_scale_dropped": ("return oracle_e4m3_to_f64(v_cache_fp8[idx]) * (double)v_scale;",
                        "return oracle_e4m3_to_f64(v_cache_fp8[idx]);"),
    "fp8_v_written_with_k_scale": ("head_dim, block_size, v_scale);", "head_dim, block_size, k_scale);"),
    "fp8_v_rows_at_key_stride": ("write_rows_e4m3(value, value_stride,", "write_rows_e4m3(value, key_stride,"),
    "mrope_index": ("double angle = pos3[i % 3] * inv_freq;", "double angle = pos3[(i / 3) % 3] * inv_freq;"),
    "fp8_fused_no_scale": ("oracle_e4m3_encode_f64(out[d] * (double)inv_scale);",
                           "oracle_e4m3_encode_f64(out[d]);"),
    "prefill_position_off_by_one": ("int64_t position = (int64_t)seq_lens[s] - n + j;",
                                    "int64_t position = (int64_t)seq_lens[s] - n + j + 1;"),
    "prefill_not_causal": ("max_blocks_per_seq, position + 1,", "max_blocks_per_seq, (int64_t)seq_lens[s],"),
    "prefill_gqa_mapping": ("num_kv_heads, h / group, head_dim, block_size, inv_sqrt_d, k_scale, v_scale,",
                            "num_kv_heads, h % num_kv_heads, head_dim, block_size, inv_sqrt_d, k_scale, v_scale,"),
    "prefill_v_with_k_scale": ("num_kv_heads, h / group, head_dim, block_size, inv_sqrt_d, k_scale, v_scale,",
                               "num_kv_heads, h / group, head_dim, block_size, inv_sqrt_d, k_scale, k_scale,"),
    "score_scale_dropped": ("scores[p - start] = (double)inv_sqrt_d * dot;", "scores[p - start] = dot;"),
    "rope_pairs_short_by_one": ("    uint32_t half = rotary_dim / 2;\n    for (uint32_t d = 0; d < head_dim; ++d) out[d] = y[d];",
                                "    uint32_t half = rotary_dim / 2 - 1;\n    for (uint32_t d = 0; d < head_dim; ++d) out[d] = y[d];"),
    "bf16_widen_shift": ("    uint32_t w = (uint32_t)bits << 16;", "    uint32_t w = (uint32_t)bits << 15;"),
    "softmax_unnormalised": ("for (uint32_t d = 0; d < head_dim; ++d) out[d] = acc[d] / denom;",
                             "for (uint32_t d = 0; d < head_dim; ++d) out[d] = acc[d];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(text.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    sys.path.insert(0, ROOT)
    import oracle
    oracle.compile_to(str(mutant_src), str(lib))
    env = dict(os.environ, PAGEDKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
