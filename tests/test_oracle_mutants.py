"""Planted mistakes: each case edits a copy of the oracle's C source in one
plausible way (a dropped term, a wrong sign or index, a transposed operand, a
wrong rounding rule), builds it on the CPU, and requires that at least one pin
in tests/pins.py catches it. The real oracle is never modified. Every mutation
keeps all memory accesses in bounds, so a mutant fails by value, not by crash."""
import os

import pytest

import oracle as O
from oracle import build as oracle_build
import pins

SRC = os.path.join(os.path.dirname(O.__file__), "oracle.c")

MUTANTS = {
    "drop_scale": ("scores[j] = scale * s;", "scores[j] = s;"),
    "lse_without_max": ("l = m + log(sum);", "l = log(sum);"),
    "normalise_by_max": ("double p = exp(scores[j] - l);", "double p = exp(scores[j] - m);"),
    "transposed_K": ("s += q[d] * K[(size_t)j * D + d];", "s += q[d] * K[(size_t)d * L + j];"),
    "gqa_map_modulo_decode": ("int hq = h * G + g;\n                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;\n                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);\n                attend_row(qd, K, V, L, D,",
                              "int hq = g * Hkv + h;\n                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;\n                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);\n                attend_row(qd, K, V, L, D,"),
    "gqa_map_modulo_window": ("int hq = h * G + g;\n                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;\n                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);\n                attend_row(qd, K + (size_t)first * D,",
                              "int hq = g * Hkv + h;\n                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;\n                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);\n                attend_row(qd, K + (size_t)first * D,"),
    "gqa_map_modulo_prefill": ("L = p + 1;                           /* causal: keys 0..p */\n        h = hq / G;",
                               "L = p + 1;                           /* causal: keys 0..p */\n        h = hq % Hkv;"),
    "gqa_map_modulo_chunked": ("L = Lk - Lq + p + 1; /* keys 0..Lk-Lq+p */\n        h = hq / G;",
                               "L = Lk - Lq + p + 1; /* keys 0..Lk-Lq+p */\n        h = hq % Hkv;"),
    "chunk_top_left_alignment": ("L = Lk - Lq + p + 1;", "L = p + 1;"),
    "window_one_key_wide": ("int first = L > window ? L - window : 0;",
                            "int first = L > window ? L - window + 1 : 0;"),
    "window_ignored": ("attend_row(qd, K + (size_t)first * D, V + (size_t)first * D, L - first,",
                       "attend_row(qd, K, V, L,"),
    "chunk_one_key_short": ("L = Lk - Lq + p + 1;", "L = Lk - Lq + p;"),
    "cache_layout_row_major_heads": ("return (((size_t)block * Hkv + h) * bs + row) * D + d;",
                                     "return (((size_t)block * bs + row) * Hkv + h) * D + d;"),
    "row_off_by_one": ("int row = j % block_size;", "int row = (j + 1) % block_size;"),
    "page_index_shift": ("int lpn = j / block_size;", "int lpn = (j + 1) / block_size;"),
    "causal_exclusive": ("L = p + 1;", "L = (p > 0) ? p : 1;"),
    "e4m3_ties_down": ("(err == best_err && (c & 1) == 0 && (best & 1) == 1)", "0"),
    "e4m3_subnormal_exponent": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "fp8_write_multiplies_scale": ("oracle_e4m3_from_f32(xk / k_scale[h])",
                                   "oracle_e4m3_from_f32(xk * k_scale[h])"),
    "fp8_dequant_ignores_scale": ("return oracle_e4m3_to_f64(((const uint8_t*)cache)[idx]) * scale_h;",
                                  "return oracle_e4m3_to_f64(((const uint8_t*)cache)[idx]);"),
    "slot_row_from_block": ("row = (int)(slot % block_size);", "row = (int)(block % block_size);"),
    "bf16_low_half": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle_build.compile_library(str(mutated), str(tmp_path / "liboracle_mutant.so"))
    with O.use_library(lib):
        failed = pins.run_all()
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_unmutated_oracle_passes_every_pin():
    assert pins.run_all() == []
