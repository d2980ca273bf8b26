"""Planted mistakes in the oracle must be caught by its pins.

Each case copies ``oracle/oracle.c``, changes one expression (a plausible slip: a
wrong GQA map, an off-by-one offset, a causal mask on the single decode query, a
dropped scale, a transposed cache index, a wrong-signed merge weight, ...),
compiles the variant into a temporary library and runs every pin on it.  At least
one pin must fail, otherwise the pins could not tell a right oracle from a wrong
one (the mutation-check idea of the llm-stack page's Model section).
"""


import pytest

import oracle as oracle_pkg
import pins

MUTATIONS = {
    "gqa_map_modulo": ("int32_t g = h / group;", "int32_t g = h % num_kv_heads;"),
    "gather_offset_off_by_one": ("int64_t offset = t % block_size;",
                                 "int64_t offset = (t + 1) % block_size;"),
    "drops_last_token": ("attend_range(o, &lse, qd, Kd, Vd, 0, len, head_dim, scale, s);",
                         "attend_range(o, &lse, qd, Kd, Vd, 0, len > 1 ? len - 1 : len, head_dim, scale, s);"),
    "causal_mask_on_decode_query": (
        "attend_range(o, &lse, qd, Kd, Vd, 0, len, head_dim, scale, s);",
        "attend_range(o, &lse, qd, Kd, Vd, 0, len > 0 ? 1 : 0, head_dim, scale, s);"),
    "missing_scale": ("s[t - t0] = scale * dot;", "s[t - t0] = dot;"),
    "cache_index_transposed": (
        "int64_t base = ((phys * num_kv_heads + g) * block_size + offset) * head_dim;",
        "int64_t base = ((phys * block_size + offset) * num_kv_heads + g) * head_dim;"),
    "merge_weight_sign": ("double w = exp(lse_part[r] - M);", "double w = exp(M - lse_part[r]);"),
    "lse_without_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "no_normalisation": ("double p = s[t - t0] / z;", "double p = s[t - t0];"),
    "write_skips_slot_zero": ("if (slot < 0) continue;", "if (slot <= 0) continue;"),
    "write_offset_swapped": ("int64_t offset = slot % block_size;",
                             "int64_t offset = (slot / block_size) % block_size;"),
    "rounding_ties_away": ("(frac == 0.5 && fmod(n, 2.0) != 0.0)", "(frac == 0.5)"),
    "widening_drops_low_bits": ("uint32_t u = ((uint32_t)bits) << 16;",
                                "uint32_t u = ((uint32_t)(bits & 0xFF80)) << 16;"),
    "rope_sine_sign": ("const float r1 = p1 - p2, r2 = p3 + p4;",
                       "const float r1 = p1 + p2, r2 = p3 - p4;"),
    "rope_wrong_partner": ("const int32_t a = neox ? i : 2 * i, b = neox ? i + half : 2 * i + 1;",
                           "const int32_t a = neox ? i : 2 * i, b = neox ? (i + 1) % half : 2 * i + 1;"),
    "rope_cos_sin_swapped": ("const float c = cs[i], s = cs[half + i];",
                             "const float c = cs[half + i], s = cs[i];"),
    "prefill_causal_off_by_one": ("attend_range(out + row, &lse, qd, Kd, Vd, 0, pos + 1, head_dim, scale, s);",
                                  "attend_range(out + row, &lse, qd, Kd, Vd, 0, pos, head_dim, scale, s);"),
    "prefill_position_from_chunk_start": ("const int32_t pos = len - n + i;",
                                          "const int32_t pos = i;"),
    "rope_k_at_position_zero": ("rope_row(krot + o, k + o, cs, head_dim, rotary_dim, neox_style);",
                                "rope_row(krot + o, k + o, cos_sin, head_dim, rotary_dim, neox_style);"),
    "rope_k_unrotated": ("rope_row(krot + o, k + o, cs, head_dim, rotary_dim, neox_style);",
                         "rope_row(krot + o, k + o, cs, head_dim, 0, neox_style);"),
    "rope_k_row_of_head_zero": (
        "rope_row(krot + o, k + o, cs, head_dim, rotary_dim, neox_style);",
        "rope_row(krot + o, k + i * num_kv_heads * (int64_t)head_dim, cs, head_dim, rotary_dim, neox_style);"),
    "q_row_of_wrong_head": (
        "qd[d] = oracle_bf16_to_double(q[((int64_t)b * num_q_heads + h) * head_dim + d]);",
        "qd[d] = oracle_bf16_to_double(q[((int64_t)b * num_q_heads + (h ^ 1)) * head_dim + d]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle_pkg._SRC).read()
    n = src.count(old)
    assert n >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle_pkg.build(str(mutated), str(tmp_path / "liboracle_mut.so"))
    o = oracle_pkg.Oracle(lib)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, RuntimeError) as e:  # noqa: PERF203
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name}"
