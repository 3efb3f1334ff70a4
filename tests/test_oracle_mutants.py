"""Plant plausible mistakes in copies of the oracle source; every copy must fail a pin.

This shows the pins are strong enough to catch a dropped term, a wrong sign
or index, a transposed operand or a wrong convention anywhere in the oracle.
The mistakes are planted in temporary copies compiled on the CPU; the
committed oracle is untouched.
"""
from pathlib import Path

import pytest

import oracle
from tests import oracle_pins

SRC = Path(oracle.__file__).resolve().parent / "ffpa_oracle.c"

MUTANTS = {
    "drop_scale": ("double x = scale * dot;", "double x = dot;"),
    "gqa_head_modulo": ("int hk = hq / group;", "int hk = hq % Hkv;"),
    "causal_offset_sign": ("i + (int64_t)Nkv - Nq", "i - (int64_t)Nkv + Nq"),
    "causal_top_left": ("i + (int64_t)Nkv - Nq", "i"),
    "lse_without_max": ("return m + log(l);", "return log(l);"),
    "mask_scaled": ("x += (double)((const float*)mask_row)[kk * mk_str];",
                    "x += scale * (double)((const float*)mask_row)[kk * mk_str];"),
    "bool_polarity": ("[kk * mk_str] == 0) x = -INFINITY;", "[kk * mk_str] != 0) x = -INFINITY;"),
    "no_normalisation": ("out[d] = acc / l;", "out[d] = acc;"),
    "keys_as_values": ("widen(vbase + (int64_t)kk * v_row_stride + d, dtype)",
                       "widen(kbase + (int64_t)kk * k_row_stride + d, dtype)"),
    "varlen_top_left": ("i + (int64_t)nk - nq", "i"),
    "fp16_exponent": ("expo - 25", "expo - 24"),
    "fp16_subnormal_exponent": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    "fp16_subnormal_implicit_bit": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)(frac | 0x400), -24);"),
    "fp16_inf_as_nan": ("mag = frac ? NAN : INFINITY;", "mag = NAN;"),
    "fp16_nan_as_inf": ("mag = frac ? NAN : INFINITY;", "mag = INFINITY;"),
    "qtype_mask_ignored": ("x += widen((const uint16_t*)mask_row + kk * mk_str, dtype);", ""),
    "masked_row_nan": ("if (m == -INFINITY) {", "if (0) {"),
    # FP8 reference
    "fp8_ties_away": ("double q = nearbyint(ldexp(a, 3 - E));", "double q = floor(ldexp(a, 3 - E) + 0.5);"),
    "fp8_subnormal_step": ("nearbyint(ldexp(a, 9));", "nearbyint(ldexp(a, 10));"),
    "fp8_exponent_bias": ("((ex + 7) << 3)", "((ex + 8) << 3)"),
    "fp8_scale_inverted": ("s = amax / 448.0f;", "s = 448.0f / amax;"),
    "fp8_no_dequant_scale": ("out[(bh * npad + r) * D + d] = e4m3_value(codes[(bh * npad + r) * D + d]) * s;",
                             "out[(bh * npad + r) * D + d] = e4m3_value(codes[(bh * npad + r) * D + d]);"),
    "fp8_mask_ignored": ("lse[r] = attend_row_f64(qrow, kb, vb, Nkv, D, scale, mask_kind, dtype, mrow, mk, limit, s,",
                         "lse[r] = attend_row_f64(qrow, kb, vb, Nkv, D, scale, ORACLE_MASK_NONE, dtype, mrow, mk, limit, s,"),
    "fp8_values_from_keys": ("acc += s[kk] * vbase[(int64_t)kk * D + d];", "acc += s[kk] * kbase[(int64_t)kk * D + d];"),
    "fp8_gqa_modulo": ("const int hk = hq / group;\n                const double* qrow",
                       "const int hk = hq % Hkv;\n                const double* qrow"),
    # backward
    "bwd_drop_delta": ("double ds = P[kk] * (dP[kk] - delta);", "double ds = P[kk] * dP[kk];"),
    "bwd_delta_sign": ("double ds = P[kk] * (dP[kk] - delta);", "double ds = P[kk] * (dP[kk] + delta);"),
    "bwd_dk_unscaled": ("dkh[(int64_t)kk * D + d] += scale * ds * widen(r.qrow + d, dtype);",
                        "dkh[(int64_t)kk * D + d] += ds * widen(r.qrow + d, dtype);"),
    "bwd_dv_with_ds": ("dvh[(int64_t)kk * D + d] += P[kk] * widen(r.dorow + d, dtype);",
                       "dvh[(int64_t)kk * D + d] += ds * widen(r.dorow + d, dtype);"),
    "bwd_dq_from_values": ("const uint16_t* krow = r.kb + (int64_t)kk * k_str[2];",
                           "const uint16_t* krow = r.vb + (int64_t)kk * v_str[2];"),
    "bwd_dp_from_keys": ("const uint16_t* vrow = vbase + (int64_t)kk * v_row_stride;",
                         "const uint16_t* vrow = kbase + (int64_t)kk * k_row_stride;"),
    "bwd_unnormalised_p": ("if (!*dead) P[kk] /= l;", ""),
    "bwd_gqa_modulo": ("int hk = hq / (Hq / Hkv);", "int hk = hq % Hkv;"),
    "bwd_causal_top_left": ("r.limit = causal ? i + (int64_t)Nkv - Nq", "r.limit = causal ? i"),
    "bwd_mask_ignored": ("dtype, scale, mask_kind, r.mrow, r.mk, r.limit, P, dP, &dead);",
                         "dtype, scale, ORACLE_MASK_NONE, r.mrow, r.mk, r.limit, P, dP, &dead);"),
    "bwd_rows_dq_unscaled": ("for (int d = 0; d < D; ++d) dqi[d] += scale * ds * widen(krow + d, dtype);",
                             "for (int d = 0; d < D; ++d) dqi[d] += ds * widen(krow + d, dtype);"),
    "bwd_rows_dv_wrong_row": ("av[d] += P[j] * widen(w.dorow + d, dtype);",
                              "av[d] += P[j] * widen(w.qrow + d, dtype);"),
    "bwd_varlen_top_left": ("int64_t limit = causal ? i + (int64_t)nk - nq : (int64_t)nk - 1;\n                    int dead;",
                            "int64_t limit = causal ? i : (int64_t)nk - 1;\n                    int dead;"),
    "bwd_varlen_key_base": ("const uint16_t* kb = k + k0 * k_str[0] + hk * k_str[1];\n            const uint16_t* vb = v + k0 * v_str[0]",
                            "const uint16_t* kb = k + q0 * k_str[0] + hk * k_str[1];\n            const uint16_t* vb = v + k0 * v_str[0]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = SRC.read_text()
    assert old in text, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    so = oracle.compile_oracle(src, tmp_path / "libmutant.so")
    mut = oracle.Oracle(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mut)
        except (AssertionError, ValueError, RuntimeError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
