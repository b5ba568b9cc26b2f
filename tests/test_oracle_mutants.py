"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant is a one-line textual change to a temporary copy of oracle.c that
keeps all memory accesses in bounds; the copy is compiled and loaded in this
process, the pins run against it, and at least one must fail.
"""

import os

import pytest

import oracle as oracle_mod
from oracle_pins import PINS

MUTANTS = {
    "gqa_modulo_map": ("const int32_t kvh = h / G;",
                       "const int32_t kvh = h % p->num_kv_heads;"),
    "no_causal_mask": ("const int32_t n = ctx + i + 1; /* keys 0 .. ctx + i */",
                       "const int32_t n = L;"),
    "mirrored_gather_offset": ("int32_t offset = j % p->block_size;",
                               "int32_t offset = (p->block_size - 1) - (j % p->block_size);"),
    "mirrored_scatter_offset": ("int64_t offset = s % block_size;",
                                "int64_t offset = (block_size - 1) - (s % block_size);"),
    "scale_dropped": ("w[j] = p->scale * dot;", "w[j] = dot;"),
    "dot_drops_last_dim": ("for (int32_t d = 0; d < D; ++d)\n            dot += qv[d]",
                           "for (int32_t d = 0; d < D - 1; ++d)\n            dot += qv[d]"),
    "unnormalised_weights": ("w[j] /= z;", "w[j] /= 1.0;"),
    "v_read_from_k_cache": ("V[(int64_t)j * D + d] = cache_value(p, p->value_cache, base + d, p->v_scale);",
                            "V[(int64_t)j * D + d] = cache_value(p, p->key_cache, base + d, p->v_scale);"),
    "fp8_exponent_bias": ("v = ldexp((double)(8 + f), e - 10);", "v = ldexp((double)(8 + f), e - 9);"),
    "fp8_subnormals_flushed": ("v = ldexp((double)f, -9);", "v = 0.0;"),
    "fp8_rounds_toward_zero": ("    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0))\n        r = fl + 1.0;",
                               "    (void)rem;"),
    "fp8_no_saturation": ("    if (a >= 448.0)\n        return sign | 0x7E;", "    if (a >= 480.0)\n        return 0x7F;"),
    "fp8_scale_divides": ("return e4m3_to_double(((const uint8_t *)cache)[idx]) * scale;",
                          "return e4m3_to_double(((const uint8_t *)cache)[idx]) / scale;"),
    "fp8_v_scale_for_k": ("K[(int64_t)j * D + d] = cache_value(p, p->key_cache, base + d, p->k_scale);",
                          "K[(int64_t)j * D + d] = cache_value(p, p->key_cache, base + d, p->v_scale);"),
    "rope_fp8_key_unrotated": ("key_cache[s * row + h * D + d] = quantize_elem(dtype, tmp[d], k_scale);",
                               "key_cache[s * row + h * D + d] = quantize_elem(dtype, key[(t * num_kv_heads + h) * D + d], k_scale);"),
    "rope_fp8_v_scale_for_k": ("key_cache[s * row + h * D + d] = quantize_elem(dtype, tmp[d], k_scale);",
                               "key_cache[s * row + h * D + d] = quantize_elem(dtype, tmp[d], v_scale);"),
    "fp8_quotient_in_double": ("float qf = xf / scale;                      /* binary32 division, correctly rounded */",
                               "double qf = (double)xf / (double)scale;"),
    "fp16_exponent_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "fp16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "copy_blocks_k_only": ("        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems, "
                           "sizeof(uint16_t) * block_elems);",
                           "        (void)value_cache;"),
    "rope_sign_flipped": ("dst[a] = double_to_elem(dtype, x1 * c - x2 * s);",
                          "dst[a] = double_to_elem(dtype, x1 * c + x2 * s);"),
    "rope_cos_sin_swapped": ("const double c = (double)cs[i], s = (double)cs[half + i];",
                             "const double s = (double)cs[i], c = (double)cs[half + i];"),
    "rope_neox_pairs_adjacent": ("const int32_t b = is_neox ? i + half : 2 * i + 1;",
                                 "const int32_t b = is_neox ? i + 1 : 2 * i + 1;"),
    "rope_key_not_rotated": ("            rotate_row(key_cache + s * row + h * D, key + (t * num_kv_heads + h) * D, "
                             "head_dim, cs, rotary_dim,\n                       is_neox, dtype);",
                             "            memcpy(key_cache + s * row + h * D, key + (t * num_kv_heads + h) * D, "
                             "sizeof(uint16_t) * (size_t)D);"),
    "round_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))", "if (frac >= 0.5)"),
    "fp16_decoded_as_bf16": ("return dtype == ORACLE_FP16 ? fp16_to_double(h) : bf16_to_double(h);",
                             "return bf16_to_double(h);"),
    "first_query_row_only": ("const uint16_t *qrow = p->q + ((int64_t)(q0 + i) * p->num_heads + h) * D;",
                             "const uint16_t *qrow = p->q + ((int64_t)(q0) * p->num_heads + h) * D;"),
    "sampled_first_row_of_request": ("int32_t i = (int32_t)(t - query_start_loc[b]);", "int32_t i = 0;"),
    "sampled_kv_head_modulo": ("gather_request(&p, b, h / G, K, V);",
                               "gather_request(&p, b, h % num_kv_heads, K, V);"),
    "drops_last_token": ("        if (s < 0)\n            continue;\n        int64_t block",
                         "        if (s < 0 || t == num_tokens - 1)\n            continue;\n        int64_t block"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    before, after = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    mutated = src.replace(before, after)
    path = os.path.join(tmp_path, f"oracle_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle_mod.compile_oracle(path, os.path.join(tmp_path, f"liboracle_{name}.so"))
    mutant = oracle_mod.Oracle(lib)
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle_mod.OracleError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
