"""Each planted mistake in a copy of the oracle must make at least one pin fail.

The mistakes are the plausible ones: a dropped term or factor, a wrong index, a
transposed operand or layout, a wrong exponent bias, a reversed copy.  Every
mutant stays inside its buffers, so running it cannot corrupt the test process.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "table_index_mod": ("table_row[t / block_size]", "table_row[t % block_size]"),
    "offset_off_by_one": ("int off = t % block_size;", "int off = (t + 1) % block_size;"),
    "dropped_scale": ("sc[t] = scale * dot;", "sc[t] = dot;"),
    "gqa_interleaved": ("const int hk = h / group;", "const int hk = h % num_kv_heads;"),
    "dropped_normalisation": ("double a = sc[t] / l;", "double a = sc[t];"),
    "dropped_last_term_of_sum": ("l += sc[t];", "if (t + 1 < L) l += sc[t];"),
    "transposed_cache_layout": (
        "return ((block * num_kv_heads + head) * block_size + offset) * (int64_t)head_dim;",
        "return ((block * block_size + offset) * num_kv_heads + head) * (int64_t)head_dim;"),
    "v_in_scores": ("dot += orc_load(q, q_dtype, qoff + d) * K[(size_t)t * head_dim + d];",
                    "dot += orc_load(q, q_dtype, qoff + d) * V[(size_t)t * head_dim + d];"),
    "k_in_output": ("o[d] += a * V[(size_t)t * head_dim + d];",
                    "o[d] += a * K[(size_t)t * head_dim + d];"),
    "query_head_as_kv_head": ("const int64_t qoff = ((int64_t)s * num_q_heads + h) * head_dim;",
                              "const int64_t qoff = ((int64_t)s * num_q_heads + hk) * head_dim;"),
    "bf16_shift": ("uint32_t w = (uint32_t)b << 16;", "uint32_t w = (uint32_t)b << 15;"),
    "f16_bias": ("ldexp((double)(frac | 0x400), expo - 25)",
                 "ldexp((double)(frac | 0x400), expo - 24)"),
    "f16_subnormal_scale": ("ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "copy_direction": ("memcpy(pool + pairs[2 * p + 1] * block_bytes, snap + p * block_bytes,",
                       "memcpy(pool + pairs[2 * p] * block_bytes, snap + p * block_bytes,"),
    "copy_sequential_not_snapshot": (
        "memcpy(pool + pairs[2 * p + 1] * block_bytes, snap + p * block_bytes,",
        "memcpy(pool + pairs[2 * p + 1] * block_bytes, pool + pairs[2 * p] * block_bytes,"),
    "reshape_wrong_block": ("int64_t blk = slot / block_size;\n",
                            "int64_t blk = (slot / block_size) ^ 1;\n"),
    "e4m3_bias": ("mag = ldexp((double)(8 + frac), expo - 10);",
                  "mag = ldexp((double)(8 + frac), expo - 9);"),
    "e4m3_subnormal": ("mag = ldexp((double)frac, -9);", "mag = ldexp((double)frac, -10);"),
    "e4m3_ties_away": ("if (d < best_d || (d == best_d && (c & 1) == 0)) {",
                       "if (d <= best_d) {"),
    "e4m3_nan_saturates": ("    if (isnan(x))\n        return 0x7f;\n",
                           "    if (isnan(x))\n        return 0x7e;\n"),
    "e4m3_scale_multiplied": ("k_cache[dst + d] = orc_f32_to_e4m3(kx / k_scale[h]);",
                              "k_cache[dst + d] = orc_f32_to_e4m3(kx * k_scale[h]);"),
    "dequant_scale_dropped": ("const double ks = k_scale ? (double)k_scale[hk] : 1.0;",
                              "const double ks = 1.0;"),
    "dequant_wrong_head_scale": ("const double vs = v_scale ? (double)v_scale[hk] : 1.0;",
                                 "const double vs = v_scale ? (double)v_scale[0] : 1.0;"),
    "chunk_top_left_causal": ("const int visible = L - n + j + 1;", "const int visible = j + 1;"),
    "chunk_excludes_own_token": ("const int visible = L - n + j + 1;",
                                 "const int visible = L - n + j;"),
    "chunk_unmasked": ("const int visible = L - n + j + 1;", "const int visible = L;"),
    "chunk_query_row_is_sequence": ("block_tables + (int64_t)s * bt_stride, (int)row, h,",
                                    "block_tables + (int64_t)s * bt_stride, s, h,"),
    "chunk_row_owner_off_by_one": ("while (query_start[s + 1] <= row)",
                                   "while (query_start[s + 1] < row)"),
    "swap_first_cache_only": ("(const char*)src[c] + pairs[2 * p] * block_bytes, (size_t)block_bytes);",
                              "(const char*)src[0] + pairs[2 * p] * block_bytes, (size_t)block_bytes);"),
    "swap_dst_is_pair_index": ("memcpy((char*)dst[c] + pairs[2 * p + 1] * block_bytes,",
                               "memcpy((char*)dst[c] + p * block_bytes,"),
    "swap_short_copy": ("(const char*)src[c] + pairs[2 * p] * block_bytes, (size_t)block_bytes);",
                        "(const char*)src[c] + pairs[2 * p] * block_bytes, (size_t)block_bytes / 2);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new), encoding="utf-8")
    so = oracle.build(str(mutant), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:
            caught.append((pin.__name__, type(e).__name__))
            break
    assert caught, f"no pin detects the planted mistake '{name}'"
