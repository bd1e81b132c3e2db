"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that the pins catch every one of them.

Each mutant is the oracle's C source with one textual change (a wrong
rounding rule, a transposed index, a dropped scale, ...), compiled into a
temporary library and run through all pins; at least one pin must fail.
"""
import os

import numpy as np
import pytest

import oracle
import oracle_pins as pins
from oracle import build as obuild
from fp8_paged_kv_attn_gb300 import inputs

MUTANTS = {
    "ties_away": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f + 1.0;"),
    "ties_down": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f;"),
    "no_saturation": ("return (uint8_t)(sign | 0x7E); /* beyond", "return (uint8_t)(sign | 0x7F); /* beyond"),
    "subnormal_bound": ("if (a < 0x1p-6) {", "if (a < 0x1p-7) {"),
    "subnormal_scale": ("round_half_even(a * 0x1p9)", "round_half_even(a * 0x1p8)"),
    "decode_sub_scale": ("ldexp((double)M, -9)", "ldexp((double)M, -10)"),
    "decode_bias": ("ldexp(8.0 + M, E - 10)", "ldexp(8.0 + M, E - 11)"),
    "decode_sign": ("return s ? -mag : mag;", "return mag;"),
    "encode_sign": ("uint8_t sign = signbit(x) ? 0x80 : 0x00;", "uint8_t sign = 0x00;"),
    "quant_mul": ("float y = x / scale;", "float y = x * scale;"),
    "quant_reciprocal": ("float y = x / scale;", "float y = x * (1.0f / scale);"),
    "append_transposed": ("int64_t dst = (((int64_t)page * H + h) * P + slot) * D + d;",
                          "int64_t dst = (((int64_t)page * P + slot) * H + h) * D + d;"),
    "append_slot": ("int slot = p % P;", "int slot = (p + 1) % P;"),
    "append_v_scale": ("oracle_quantise(v_new[src], v_scale)", "oracle_quantise(v_new[src], k_scale)"),
    "check_floor_pages": ("int n_pages = (L + page_size - 1) / page_size;\n            for",
                          "int n_pages = L / page_size;\n            for"),
    "check_no_range": ("if (page < 0 || page >= num_pages) { bad = 1; continue; }",
                       "if (page < 0 || page >= num_pages) { continue; }"),
    "check_no_len": ("if (L < 0 || (int64_t)L > (int64_t)MP * page_size) {\n            bad = 1;",
                     "if (L < 0 || (int64_t)L > (int64_t)MP * page_size) {\n            bad = 0;"),
    "attn_head_map": ("int kvh = h / g;", "int kvh = h % H;"),
    "attn_no_kscale": ("(cached_value(kv_dtype, k_pool, base + d) * k_scale)",
                       "(cached_value(kv_dtype, k_pool, base + d))"),
    "attn_no_vscale": ("(cached_value(kv_dtype, v_pool, base + d) * v_scale)",
                       "(cached_value(kv_dtype, v_pool, base + d))"),
    "attn_no_smscale": ("s *= sm_scale;", "s *= 1.0;"),
    "attn_v_from_k": ("acc[d] += w * (cached_value(kv_dtype, v_pool,", "acc[d] += w * (cached_value(kv_dtype, k_pool,"),
    "attn_drop_last": ("        double w = exp(logits[j] - m);", "        if (j == L - 1) continue;\n        double w = exp(logits[j] - m);"),
    "attn_ignore_abort": ("if (abort_mask && abort_mask[b]) return 0;", "(void)abort_mask;"),
    "attn_no_normalise": ("o[d] = (float)(acc[d] / denom);", "o[d] = (float)(acc[d]);"),
    "attn_slot": ("int64_t base = (((int64_t)page * H + kvh) * P + j % P) * D;\n        double s",
                  "int64_t base = (((int64_t)page * H + kvh) * P + (j + 1) % P) * D;\n        double s"),
    "pages_bump_on_release": ("free_stack[count++] = *entry;\n                *entry = -1;",
                              "free_stack[count++] = *entry;\n                page_tags[*entry] += 1u;\n                *entry = -1;"),
    "pages_no_bump": ("page_tags[page] += 1u;", "page_tags[page] += 0u;"),
    "pages_pop_order": ("int page = free_stack[--count];",
                        "int page = free_stack[count - n + k];\n            if (k == n - 1) count -= n;"),
    "pages_keep_entry": ("                *entry = -1;\n", "\n"),
    "pages_no_stop": ("if (stopped || n > count) { stopped = 1;", "if (n > count) { stopped = 1;"),
    "pages_old_tag": ("expected_tags[(int64_t)b * MP + first + k] = page_tags[page];",
                      "expected_tags[(int64_t)b * MP + first + k] = page_tags[page] - 1u;"),
    "pages_partial_release": ("    if (rel_err) {\n        err |= rel_err;\n    } else {",
                              "    err |= rel_err;\n    {"),
    "pages_first_ignored": ("block_table[(int64_t)b * MP + first + k] = page;",
                            "block_table[(int64_t)b * MP + k] = page;"),
    "wq_nibble_order": ("int nib = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                        "int nib = (k % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "wq_unsigned": ("return nib >= 8 ? nib - 16 : nib;", "return nib - 8;"),
    "handoff_src_slot": ("int slot = (int)(p % src_P);", "int slot = (int)(p % dst_P);"),
    "handoff_first_ignored": ("int64_t f = first ? first[b] : 0;", "int64_t f = 0;"),
    "handoff_src_page_unchecked": ("if (sp < 0 || sp >= src_pages) { err |= ORACLE_ERR_PAGE; continue; }",
                                   "if (sp < 0) { err |= ORACLE_ERR_PAGE; continue; }"),
    "wq_group": ("(double)bf16_to_float(s[k / group]);", "(double)bf16_to_float(s[k / 64]);"),
    "wq_no_e4m3_scale": ("wv = oracle_e4m3_decode(row[k]) * (double)s[n];",
                         "wv = oracle_e4m3_decode(row[k]);"),
    "attn_bf16_scaled": ("double ks = (kv_dtype == ORACLE_KV_E4M3) ? (double)k_scale : 1.0;",
                         "double ks = (double)k_scale;"),
}


def run_all_pins():
    """Run every pin; return the names of those that failed."""
    small = inputs.uniform("u", 11, B=3, ctx=70, Hq=8, Hkv=2, D=64, P=16, outlier_frac=0.01)
    checks = [
        ("decode_all_codes", lambda: pins.pin_decode_all_codes(oracle)),
        ("decode_structure", lambda: pins.pin_decode_structure(oracle)),
        ("encode_roundtrip", lambda: pins.pin_encode_roundtrip(oracle)),
        ("encode_vs_torch", lambda: pins.pin_encode_vs_torch(oracle)),
        ("encode_brute", lambda: pins.pin_encode_brute_force(oracle)),
        ("encode_special", lambda: pins.pin_encode_special(oracle)),
        ("quantise_exhaustive", lambda: pins.pin_quantise_exhaustive(oracle)),
        ("append_slots", lambda: pins.pin_append_slots(oracle, small)),
        ("append_bf16", lambda: pins.pin_append_bf16_copy(oracle, small)),
        ("append_errors", lambda: pins.pin_append_errors(oracle)),
        ("check_injected", lambda: pins.pin_check_injected(
            oracle, inputs.integrity(seed=21, B=64, lo=16, hi=600, stale_frac=0.1))),
        ("check_edges", lambda: pins.pin_check_edges(oracle)),
        ("attn_sdpa", lambda: pins.pin_attn_vs_sdpa(oracle, small)),
        ("attn_sdpa_bf16", lambda: pins.pin_attn_vs_sdpa(oracle, small, kv_dtype=oracle.KV_BF16)),
        ("attn_one_token", lambda: pins.pin_attn_one_token(oracle)),
        ("attn_equal_keys", lambda: pins.pin_attn_equal_keys(oracle)),
        ("attn_abort", lambda: pins.pin_attn_abort_and_errors(oracle)),
        ("int4_nibbles", lambda: pins.pin_int4_nibbles(oracle)),
        ("handoff", lambda: pins.pin_handoff_vs_torch(oracle)),
        ("wq_vs_numpy", lambda: pins.pin_wq_vs_numpy(oracle)),
        ("wq_single", lambda: pins.pin_wq_single_weight(oracle)),
        ("wq_wide_range_x", lambda: pins.pin_wq_wide_range_x(oracle)),
        ("pages_golden", lambda: pins.pin_pages_golden(oracle)),
        ("pages_invariants", lambda: pins.pin_pages_invariants(oracle, n_ops=30)),
        ("pages_overflow", lambda: pins.pin_pages_overflow_and_state(oracle)),
    ]
    failed = []
    for name, fn in checks:
        try:
            with np.errstate(all="ignore"):
                fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert run_all_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    find, repl = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(find) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(find, repl))
    so = obuild.compile_to(str(path), str(tmp_path / f"lib{name}.so"))
    with oracle.use_library(so):
        failed = run_all_pins()
    assert failed, f"no pin caught mutant {name}"
    os.remove(so)
