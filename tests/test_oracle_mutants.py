"""Planted mistakes: each altered copy of the oracle must fail at least one pin.

Every mutant below is a plausible slip (a dropped term, a wrong sign or index,
a transposed operand, a skipped step) planted in a temporary copy of
oracle.c, compiled with gcc on the CPU.  The pins in test_oracle_pins.py are
then run against the mutant; the test passes only if some pin catches it.
"""
import inspect

import pytest

import oracle
import test_oracle_fp8 as fp8_pins
import test_oracle_pins as pins

MUTANTS = {
    "pool_drop_last_term": ("for (int j = 0; j < P; ++j) {", "for (int j = 0; j < P - 1; ++j) {"),
    "pool_wrong_token_index": ("(P * g + j) * (int64_t)d + i", "(g + j) * (int64_t)d + i"),
    "pool_weights_reversed": ("double aj = (double)alpha[j];", "double aj = (double)alpha[P - 1 - j];"),
    "pool_ties_away_from_zero": ("if (half && (sticky || (r & 1u)))", "if (half)"),
    "pool_sticky_bits_ignored": ("if (half && (sticky || (r & 1u)))", "if (half && (r & 1u))"),
    "pool_negation_drops_carry": ("carry = carry && a->w[i] == 0;", "carry = 0;"),
    "pool_nine_significant_bits": ("int qe = top + WIDE_E0 - 7;", "int qe = top + WIDE_E0 - 8;"),
    "bf16_truncates": ("double r = rint(ldexp(a, -qe));", "double r = floor(ldexp(a, -qe));"),
    "score_no_relu": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "score_wrong_head_weight": ("s += (double)wt[h] * relu;", "s += (double)wt[0] * relu;"),
    "score_query_transposed": ("dot += bf16_value(qt[h * d + i]) * bf16_value(kg[i]);",
                               "dot += bf16_value(qt[i * H_i + h]) * bf16_value(kg[i]);"),
    "mask_off_by_one": ("int64_t m = (p + 1) / P;", "int64_t m = p / P + 1;"),
    "select_ascending": ("    if (a->s > b->s)\n        return -1;\n    if (a->s < b->s)\n        return 1;",
                         "    if (a->s < b->s)\n        return -1;\n    if (a->s > b->s)\n        return 1;"),
    "select_ties_to_higher_index": ("return (a->g < b->g) ? -1 : (a->g > b->g);",
                                    "return (a->g > b->g) ? -1 : (a->g < b->g);"),
    "select_unsorted_output": ("qsort(out, (size_t)m, sizeof(int32_t), by_index_asc);", ""),
    "attn_no_scale": ("z[j] = scale * dot;", "z[j] = dot;"),
    "attn_unnormalised": ("oh[i] = oracle_bf16_from_double(o[i] / l);",
                          "oh[i] = oracle_bf16_from_double(o[i]);"),
    "attn_values_from_keys": ("const uint16_t *vj = V + b * sV_b + tok[j] * d_v;",
                              "const uint16_t *vj = K + b * sK_b + tok[j] * d_qk;"),
    "attn_lse_sign": ("*lh = (float)(m + log(l));", "*lh = (float)(m - log(l));"),
}


# the quantized legs (e4m3 and INT8 codes, per-row scales, FP8 score, FP8 and
# INT8 K/V attention), caught by test_oracle_fp8
FP8_MUTANTS = {
    "i8_ties_to_odd": ("(d == bd && c % 2 == 0)", "(d == bd && c % 2 == 1)"),
    "i8_scale_divisor": ("const float sc = (float)(amax / 127.0);",
                         "const float sc = (float)(amax / 128.0);"),
    "i8_sign_lost": ("return (int8_t)(x < 0.0 ? -best : best);", "return (int8_t)best;"),
    "i8kv_value_scale_dropped": ("acc[i] += wj * oracle_i8_value(vr[i], vscale);",
                                 "acc[i] += wj * oracle_i8_value(vr[i], 1.0f);"),
    "i8kv_key_scale_dropped": ("qk += bf16_value(qv[i]) * oracle_i8_value(kr[i], kscale);",
                               "qk += bf16_value(qv[i]) * oracle_i8_value(kr[i], 1.0f);"),
    "i8kv_unnormalised": ("ov[i] = oracle_bf16_from_double(acc[i] / denom);",
                          "ov[i] = oracle_bf16_from_double(acc[i]);"),
    "i8kv_no_softmax_scale": ("zs[j] = scale * qk;", "zs[j] = qk;"),
    "e4m3_exponent_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_ties_to_odd": ("(d == bd && (c & 1) == 0)", "(d == bd && (c & 1) == 1)"),
    "e4m3_no_saturation": ("if (a >= 448.0) return sign | 0x7E;",
                           "if (a >= 448.0) return sign | 0x7F;"),
    "e4m3_sign_lost": ("    return sign | best;", "    return best;"),
    "quantize_scale_not_applied": ("oracle_e4m3_from_double(bf16_value(xr[i]) / (double)sc)",
                                   "oracle_e4m3_from_double(bf16_value(xr[i]))"),
    "kv8_value_scale_dropped": ("o[i] += p * (oracle_e4m3_value(vj[i]) * sv);",
                                "o[i] += p * oracle_e4m3_value(vj[i]);"),
    "kv8_key_scale_dropped": ("dot += bf16_value(qh[i]) * (oracle_e4m3_value(kj[i]) * sk);",
                              "dot += bf16_value(qh[i]) * oracle_e4m3_value(kj[i]);"),
    "kv8_scales_swapped": ("const double sv = (double)vs[b * svs_b + tok[j]];",
                           "const double sv = (double)ks[b * sks_b + tok[j]];"),
    "fp8_score_drops_key_scale": ("dot *= (double)sq[qr] * (double)sk[kr];",
                                  "dot *= (double)sq[qr];"),
    "fp8_score_no_relu": ("s += (double)w_head[qr] * (dot > 0.0 ? dot : 0.0);",
                          "s += (double)w_head[qr] * dot;"),
}


def _fp8_pin_calls():
    calls = [(f"hand_{x}", lambda x=x, c=c: fp8_pins.test_e4m3_hand_encodings(x, c))
             for x, c in fp8_pins.HAND]
    for name, fn in inspect.getmembers(fp8_pins, inspect.isfunction):
        if name.startswith("test_") and not inspect.signature(fn).parameters:
            calls.append((name, fn))
    return calls


@pytest.mark.parametrize("mutant", sorted(FP8_MUTANTS))
def test_fp8_pins_catch_planted_mistake(mutant, tmp_path):
    old, new = FP8_MUTANTS[mutant]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor not unique/absent: {mutant}"
    so = str(tmp_path / f"oracle_{mutant}.so")
    oracle.compile_variant(src.replace(old, new), so)
    caught = []
    with oracle.use_library(so):
        for name, call in _fp8_pin_calls():
            try:
                call()
            except Exception:
                caught.append(name)
    assert caught, f"no FP8 pin caught mutant {mutant}"


def test_unmutated_copy_passes_every_fp8_pin(tmp_path):
    so = str(tmp_path / "oracle_copy_fp8.so")
    oracle.compile_variant(oracle.source(), so)
    with oracle.use_library(so):
        for name, call in _fp8_pin_calls():
            call()


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = inspect.signature(fn).parameters
        if "j" in params:
            calls.append((name, lambda fn=fn: fn(1)))
        elif not params:
            calls.append((name, fn))
    return calls


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor not unique/absent: {mutant}"
    so = str(tmp_path / f"oracle_{mutant}.so")
    oracle.compile_variant(src.replace(old, new), so)
    caught = []
    with oracle.use_library(so):
        for name, call in _pin_calls():
            try:
                call()
            except Exception:
                caught.append(name)
    assert caught, f"no pin caught mutant {mutant}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    so = str(tmp_path / "oracle_copy.so")
    oracle.compile_variant(oracle.source(), so)
    with oracle.use_library(so):
        for name, call in _pin_calls():
            call()
