"""Plant plausible mistakes in copies of the oracle source; every copy must fail a pin.

This shows the pins are strong enough to catch a dropped term, a wrong sign
or index, a transposed operand or a wrong convention anywhere in the oracle.
The mistakes are planted in temporary copies compiled on the CPU; the
committed oracle is untouched.
"""
import shutil
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
    "qtype_mask_ignored": ("x += widen((const uint16_t*)mask_row + kk * mk_str, dtype);", ""),
    "masked_row_nan": ("if (m == -INFINITY) {", "if (0) {"),
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
