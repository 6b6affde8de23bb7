"""Planted mistakes in copies of the oracle must each fail at least one pin (no GPU).

Each mutant is a plausible slip -- a wrong index, a dropped term, a wrong exponent bias, a
swapped operand -- applied as a text edit to a temporary copy of ``oracle/pa_oracle.c``. The
real oracle is never modified. If a mutant survives every pin, the pins are too weak.
"""
import os
import shutil

import pytest

import oracle
from pins import ALL_PINS

# (name, original text, planted text, occurrences)
MUTANTS = [
    ('gqa_group_by_modulo', 'const int g = h / group;', 'const int g = h % num_kv_heads;', 2),
    ('slot_off_by_one', 'const int slot = t % block_size; /* slot', 'const int slot = (t + 1) % block_size; /* slot', 1),
    ('table_row_ignored', 'block_tables[(size_t)s * max_blocks_per_seq + j]', 'block_tables[j]', 1),
    ('heads_inside_slots', '(((size_t)phys * num_kv_heads + g) * block_size + slot) * head_dim', '(((size_t)phys * block_size + slot) * num_kv_heads + g) * head_dim', 1),
    ('scale_dropped', 'score[t] = scale * dot;', 'score[t] = dot;', 2),
    ('no_max_shift', 'score[t] = exp(score[t] - max_score);', 'score[t] = exp(score[t]);', 2),
    ('no_normalisation', 'o[d] = acc / denom;', 'o[d] = acc;', 2),
    ('k_scale_dropped', 'element(k_pool, first + d, kv_dtype) * k_scale', 'element(k_pool, first + d, kv_dtype)', 1),
    ('v_scale_dropped', 'element(v_pool, first + d, kv_dtype) * v_scale', 'element(v_pool, first + d, kv_dtype)', 1),
    ('v_read_from_k_pool', 'element(v_pool, first + d, kv_dtype)', 'element(k_pool, first + d, kv_dtype)', 2),
    ('drops_newest_token', 'for (int t = 0; t < L; ++t) {\n        double dot', 'for (int t = 0; t < L - 1; ++t) {\n        double dot', 1),
    ('e4m3_bias_8', 'e - 7 - 3', 'e - 8 - 3', 1),
    ('e4m3_subnormal_as_normal', 'mag = ldexp((double)f, -6 - 3);', 'mag = ldexp((double)(8 + f), -7 - 3);', 1),
    ('e4m3_nan_as_number', 'if (e == 15 && f == 7) {', 'if (0) {', 1),
    ('bf16_bias_126', 'e - 127 - 7', 'e - 126 - 7', 1),
    ('f16_subnormal_scale', 'mag = ldexp((double)f, -24);', 'mag = ldexp((double)f, -25);', 1),
    ('f16_sign_ignored', 'return sign ? -mag : mag;\n}\n\n/* bfloat16', 'return mag;\n}\n\n/* bfloat16', 1),
    ('write_slot_zero', 'const int64_t slot = sigma % block_size;', 'const int64_t slot = 0;', 2),
    ('write_v_from_k', 'memcpy((uint8_t*)v_pool + dst, (const uint8_t*)v + src, row);', 'memcpy((uint8_t*)v_pool + dst, (const uint8_t*)k + src, row);', 1),
    ('write_head_stride_dropped', 'const size_t src = ((size_t)t * num_kv_heads + h) * row;', 'const size_t src = (size_t)t * row;', 1),
    ('copy_forgets_v', 'memcpy((uint8_t*)v_pools[l] + (size_t)dst * block_bytes, keep + block_bytes, block_bytes);', '', 1),
    ('copy_only_first_layer', 'for (int l = 0; l < num_layers; ++l) {\n      const uint8_t* keep', 'for (int l = 0; l < 1; ++l) {\n      const uint8_t* keep', 1),
    ('swap_k_v_same_slot', '(((size_t)i * num_layers + l) * 2 + 1) * block_bytes', '(((size_t)i * num_layers + l) * 2 + 0) * block_bytes', 1),
    ('swap_layer_major', '(((size_t)i * num_layers + l) * 2', '(((size_t)l * n + i) * 2', 2),
    ('encode_truncates', 'if (r > 0.5 || (r == 0.5 && (q & 1u))) ++q;', '', 1),
    ('encode_ties_away', '(r == 0.5 && (q & 1u))', '(r == 0.5)', 1),
    ('encode_no_saturation', 'if (a >= 448.0) return sign | 0x7E;', 'if (a >= 480.0) return sign | 0x7F;', 1),
    ('encode_bias_8', '((E + 7) << 3)', '((E + 8) << 3)', 1),
    ('encode_subnormal_step', 'round_half_even(ldexp(a, 9))', 'round_half_even(ldexp(a, 8))', 1),
    ('encode_sign_dropped', 'return sign | (uint8_t)(((E + 7) << 3) | q);', 'return (uint8_t)(((E + 7) << 3) | q);', 1),
    ('quantise_by_scale_not_inverse', '* (double)k_inv', '* (double)k_scale', 1),
    ('quantise_v_with_k_inverse', '* (double)v_inv', '* (double)k_inv', 1),
    ('prefill_sees_future', 't <= last', 't < L', 3),
    ('prefill_position_from_chunk_start', 'const int last = L - n + i;', 'const int last = i;', 1),
    ('prefill_excludes_itself', 'const int last = L - n + i;', 'const int last = L - n + i - 1;', 1),
    ('prefill_scale_dropped', '          score[t] = scale * dot;', '          score[t] = dot;', 1),
    ('prefill_v_from_k', 'v_scale * element(v_pool, first + d, kv_dtype);', 'v_scale * element(k_pool, first + d, kv_dtype);', 1),
    ('prefill_k_scale_dropped', 'K[(size_t)t * head_dim + d] = k_scale * element', 'K[(size_t)t * head_dim + d] = element', 1),
    ('prefill_v_scale_dropped', 'V[(size_t)t * head_dim + d] = v_scale * element', 'V[(size_t)t * head_dim + d] = element', 1),
    ('prefill_v_with_k_scale', 'V[(size_t)t * head_dim + d] = v_scale * element', 'V[(size_t)t * head_dim + d] = k_scale * element', 1),
    ('prefill_query_read_as_kv_dtype', 'dot += element(q, qoff + d, q_dtype) * K[(size_t)t * head_dim + d];\n          score[t]', 'dot += element(q, qoff + d, kv_dtype) * K[(size_t)t * head_dim + d];\n          score[t]', 1),
    ('prefill_query_row_of_chunk_start', 'const size_t qoff = ((size_t)(q_starts[s] + i) * num_q_heads + h) * head_dim;', 'const size_t qoff = ((size_t)(q_starts[s]) * num_q_heads + h) * head_dim;', 1),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, count):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == count, f"mutation site for {name} not found; update the mutant"
    mutated = tmp_path / "pa_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(str(mutated), str(tmp_path / f"lib_{name}.so"), openmp=False)
    orc = oracle.load(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as exc:  # AssertionError, or a crash-free error from garbage values
            caught.append(f"{pin.__name__}: {type(exc).__name__}")
    assert caught, f"mutant {name} survived every pin"
