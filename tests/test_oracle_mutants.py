"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source (a dropped term, a wrong sign, a wrong index, a wrong
tie rule, a transposed operand), builds it on the CPU, swaps it in for the
real oracle, and requires at least one pin to fail. The real oracle is
restored afterwards."""
import ctypes as C
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moeperm_oracle.c")

# (name, original text, planted mistake, pin tests that must catch it)
MUTANTS = [
    ("tie_away_from_zero", "else pick = (c & 1) ? c + 1 : c;", "else pick = c + 1;",
     ["test_e4m3_encode_matches_library_rne"]),
    ("swapped_distances", "double dl = a - vc, du = vn - a;", "double du = a - vc, dl = vn - a;",
     ["test_e4m3_encode_matches_library_rne"]),
    ("wrong_fp8_max", "int k = (int)ceil(log2(a / 448.0));               /* first guess */\n"
     "  while (ldexp(448.0, k) < a) ++k;                   /* exact fix-ups */\n"
     "  while (ldexp(448.0, k - 1) >= a) --k;",
     "int k = (int)ceil(log2(a / 240.0));\n  while (ldexp(240.0, k) < a) ++k;\n"
     "  while (ldexp(240.0, k - 1) >= a) --k;",
     ["test_group_exponent_closed_forms", "test_group_exponent_interval_exact"]),
    ("scale_bias", "ebytes[gi] = (uint8_t)(e + 127);", "ebytes[gi] = (uint8_t)(e + 128);",
     ["test_quant_row_against_library", "test_quant_row_zero_group"]),
    ("eps_changed", "const float eps = 1e-10f;\n  double a", "const float eps = 1e-12f;\n  double a",
     ["test_group_exponent_closed_forms", "test_quant_row_zero_group"]),
    ("scale_sign", "q[h] = ref_e4m3_encode(ldexp(bf16_value(x[h]), -e));",
     "q[h] = ref_e4m3_encode(ldexp(bf16_value(x[h]), e));", ["test_quant_row_against_library"]),
    ("group_index_off", "double a = fabs(bf16_value(x[h]));",
     "double a = fabs(bf16_value(x[h < H - 1 ? h + 1 : h]));", ["test_quant_row_against_library"]),
    ("packed_word_transposed", "int64_t word = b * (int64_t)g4_of(G) * ld + (int64_t)(gi / 4) * ld + r;",
     "int64_t word = b * (int64_t)g4_of(G) * ld + (int64_t)(gi / 4) + r * g4_of(G);",
     ["test_dispatch_compact_invariants_random"]),
    ("unaligned_segments", "acc += align_up(counts[e], block_e);", "acc += counts[e];",
     ["test_dispatch_compact_invariants_random"]),
    ("bound_drops_term", "return block_e * (n + (A - n) / block_e);", "return block_e * n;",
     ["test_compact_bound_brute_force"]),
    ("masked_rule_flipped", "return (E > L && L <= 32) ? 1 : 0;", "return (E >= L && L <= 32) ? 1 : 0;",
     ["test_masked_rule_truth_table"]),
    ("combine_drops_first_slot", "for (int32_t k = 0; k < K; ++k) {\n        int32_t row = src2dst[(int64_t)t * K + k];\n        if (row < 0) continue;\n        double wk",
     "for (int32_t k = 1; k < K; ++k) {\n        int32_t row = src2dst[(int64_t)t * K + k];\n        if (row < 0) continue;\n        double wk",
     ["test_combine_f64_against_numpy"]),
    ("requant_ratio_inverted", "float r = (S > 0.0f) ? s_tok[t] / S : 0.0f;",
     "float r = (S > 0.0f) ? S / s_tok[t] : 0.0f;", ["test_requant_against_library"]),
    ("bf16_truncates", "u += 0x7FFFu + lsb;", "u += 0u * lsb;", ["test_bf16_rne_matches_library"]),
    ("slab_row_index", "int64_t src = start[e] + j, dst = (int64_t)e * cap + j;",
     "int64_t src = start[e] + j, dst = (int64_t)e * cap + (cap - 1 - j);", ["test_repack_roundtrip"]),
    ("masked_m_unclamped", "masked_m[e] = counts[e] < cap ? counts[e] : cap;", "masked_m[e] = counts[e];",
     ["test_dispatch_masked_overflow"]),
    ("rank_order_reversed", "for (int64_t a = 0; a < (int64_t)T * K; ++a) {\n    int32_t t = (int32_t)(a / K);",
     "for (int64_t a = (int64_t)T * K - 1; a >= 0; --a) {\n    int32_t t = (int32_t)(a / K);",
     ["test_dispatch_compact_invariants_random", "test_dispatch_compact_exhaustive_tiny"]),
    ("m_indices_tail_filled", "for (int64_t r = 0; r < bound; ++r) m_indices[r] = -1;",
     "for (int64_t r = 0; r < bound; ++r) m_indices[r] = L - 1;",
     ["test_dispatch_compact_invariants_random", "test_dispatch_compact_exhaustive_tiny"]),
    ("masked_psum_unaligned", "int64_t seg_start = align_up(prev_end, psum_align);",
     "int64_t seg_start = prev_end;", ["test_dispatch_masked_psum_equals_compact_layout"]),
    ("masked_psum_unclamped", "psum[e] = (int32_t)(seg_start + masked_m[e]);",
     "psum[e] = (int32_t)(seg_start + counts[e]);",
     ["test_dispatch_masked_psum_overflow_follows_masked_m"]),
    ("overflow_flag_off_by_one", "if (counts[e] > cap) st |= REF_ST_OVERFLOW;",
     "if (counts[e] > cap + 1) st |= REF_ST_OVERFLOW;", ["test_dispatch_masked_overflow"]),
    # widened rows: OCP-MX exponent, plain fp32 scales, e8m0 / amax requant, weighted repack
    ("mx_emax_off_by_one", "  int X = k - 8;", "  int X = k - 7;",
     ["test_mx_exponent_closed_forms_and_interval", "test_quant_row_mx_against_library"]),
    ("f32_scale_divisor", "      float sc = a / 448.0f;", "      float sc = a / 240.0f;",
     ["test_quant_row_f32_against_library"]),
    ("f32_quotient_inverted", "        float v = (float)bf16_value(x[h]) / sc;",
     "        float v = (float)bf16_value(x[h]) * sc;", ["test_quant_row_f32_against_library"]),
    ("requant_amax_drops_token_scale", "      v = s[t] * (float)amax;", "      v = (float)amax;",
     ["test_requant_ex_amax_mode_against_library"]),
    ("requant_amax_divisor", "  if (mode == 1) S = S / 448.0f;", "  if (mode == 1) S = S / 240.0f;",
     ["test_requant_ex_amax_mode_against_library"]),
    ("e8m0_decode_bias", "(int)((const uint8_t*)s_tok)[t] - 127);", "(int)((const uint8_t*)s_tok)[t] - 128);",
     ["test_requant_ex_ue8m0_scales_are_exact_powers"]),
    ("repack_weight_ignored", "d16[h] = ref_bf16_rne(wr * (float)bf16_value(s16[h]));",
     "d16[h] = ref_bf16_rne((float)bf16_value(s16[h]));", ["test_repack_weighted_rows"]),
]


def build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    hdr = os.path.join(os.path.dirname(SRC), "moeperm_oracle.h")
    (tmp_path / "moeperm_oracle.h").write_text(open(hdr).read())
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(path), "-lm"], check=True)
    lib = C.CDLL(str(so))
    oracle._declare(lib)
    return lib


def run_pin(name):
    fn = getattr(pins, name)
    import inspect
    params = inspect.signature(fn).parameters
    if "counts" in params:          # parametrised repack pin: run one representative case
        fn(oracle, [3, 0, 5, 1], "bf16")
    elif "align" in params:
        fn(oracle, 128)
    elif "fmt" in params:
        fn(oracle, "packed")
    elif "g" in params:
        fn(oracle, 128, 640)
    elif "H" in params:
        fn(oracle, 224)
    else:
        fn(oracle)


@pytest.mark.parametrize("mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(ref, tmp_path, mut):
    name, old, new, catchers = mut
    real = oracle.lib()
    mutant = build_mutant(tmp_path, name, old, new)
    oracle._lib = mutant
    try:
        caught = []
        for pin in catchers:
            try:
                run_pin(pin)
            except AssertionError:
                caught.append(pin)
        assert caught, f"mutant {name} passed the pins {catchers}"
    finally:
        oracle._lib = real
