"""Planted mistakes in (copies of) the oracle must each fail at least one pin.

Each mutant is the oracle's C source with one plausible slip applied as a text
substitution (a wrong index, a dropped term, a wrong sign, a transposed
layout, a wrong exponent bias), compiled with gcc into a temporary library.
The mistake is planted in the oracle on the CPU; nothing here touches a GPU.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_CHECKS

MUTANTS = {
    "block_index_mod": ("p = block_tables[(size_t)i * MB + t / bs];\n        int off = t % bs;\n        if (p < 0",
                        "p = block_tables[(size_t)i * MB + t % bs];\n        int off = t % bs;\n        if (p < 0"),
    "row_offset_div": ("int off = t % bs;\n        if (p < 0", "int off = t / bs;\n        if (p < 0"),
    "gqa_mod_mapping": ("int g = h / G;", "int g = h % Hkv;"),
    "dropped_scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "softmax_sign": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "dropped_normalisation": ("for (int d = 0; d < D; ++d) out[d] /= Z;", ""),
    "cache_layout_transposed": ("k_cache + (((size_t)p * Hkv + g) * bs + off) * D;",
                                "k_cache + (((size_t)g * NB + p) * bs + off) * D;"),
    "v_uses_k": ("v_cache + (((size_t)p * Hkv + g) * bs + off) * D;",
                 "k_cache + (((size_t)p * Hkv + g) * bs + off) * D;"),
    "half_bias": ("e - 25", "e - 24"),
    "half_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16_bias": ("e - 134", "e - 133"),
    "last_token_dropped": ("for (int t = 0; t < L; ++t) {\n        int p = block_tables[(size_t)i * MB + t / bs];\n        int off = t % bs;\n        const",
                           "for (int t = 0; t < L - 1; ++t) {\n        int p = block_tables[(size_t)i * MB + t / bs];\n        int off = t % bs;\n        const"),
    "append_offset": ("int blk = s / bs, off = s % bs;", "int blk = s / bs, off = s % bs ^ 1;"),
    "append_negative_slot_written": ("if (s < 0) continue;", "if (s < 0) s = 0;"),
    "q_head_shared": ("q + ((size_t)i * Hq + h) * D;", "q + ((size_t)i * Hq + h / (Hq / Hkv)) * D;"),
    "copy_swapped_pair": ("int s = pairs[2 * i], d = pairs[2 * i + 1];",
                          "int d = pairs[2 * i], s = pairs[2 * i + 1];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(mutated), str(tmp_path / "libmutant.so")))
    failed = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
