"""CPU tests: the float64 oracle against its pins, and planted mistakes in
mutated copies of the oracle that the pins must catch."""
import os
import shutil
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


# Each mutant replaces one exact fragment of the oracle source with a plausible mistake.
MUTANTS = {
    "dropped_rope_in_scores": ("for (d = 0; d < ORACLE_QK_DIM; ++d) acc +=", "for (d = 0; d < ORACLE_V_DIM; ++d) acc +="),
    "value_from_wrong_offset": ("out[j] += w * kv_value(kv, row, j, mode, kv_scale)",
                                "out[j] += w * kv_value(kv, row, j + 64, mode, kv_scale)"),
    "e4m3_exponent_bias": ("ldexp(8.0 + (double)m, e - 10)", "ldexp(8.0 + (double)m, e - 9)"),
    "e4m3_subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_decode_sign": ("return s ? -v : v;", "return v;"),
    "encode_truncates": ("if (a - vlo < vhi - a) return", "if (1) return"),
    "encode_ties_up": ("((lo & 1) ? lo + 1 : lo)", "(lo + 1)"),
    "encode_overflow_nan": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);",
                            "if (a >= 464.0) return (uint8_t)(sign | 0x7F);"),
    "kv_scale_dropped": ("[row * ORACLE_QK_DIM + d]) * kv_scale;", "[row * ORACLE_QK_DIM + d]);"),
    "q_cast_skipped": ("if (mode == 1) v = oracle_e4m3_decode(oracle_e4m3_encode(v));", ""),
    "missing_normalisation": ("double w = s[t] / z;", "double w = s[t];"),
    "missing_sm_scale": ("s[t] = sm_scale * acc;", "s[t] = acc;"),
    "wrong_head": ("(q_row * ORACLE_HEADS + h) * ORACLE_QK_DIM", "(q_row * ORACLE_HEADS + 0) * ORACLE_QK_DIM"),
    "causal_off_by_one": ("int64_t n = causal ? L - qb + j + 1 : L;", "int64_t n = causal ? L - qb + j : L;"),
    "query_row_of_sequence": ("(int)row_seq[r], r, h, 0, row_len[r]", "(int)row_seq[r], row_seq[r], h, 0, row_len[r]"),
    "indices_ignored": ("return (int64_t)kv_indices[page_base + t / page_size] * page_size + t % page_size;",
                        "return page_base * page_size + t;"),
    "page_offset_dropped": ("* page_size + t % page_size;", "* page_size;"),
    "last_page_len_ignored": ("return (pages - 1) * page_size + last;", "return pages * page_size;"),
    "lse_missing_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "combine_unnormalised": ("double w = exp(part_lse[s * ORACLE_HEADS + h] - m) / z;",
                             "double w = exp(part_lse[s * ORACLE_HEADS + h] - m);"),
    "bf16_decode_shift": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    old, new = MUTANTS[name]
    assert old in src, f"mutation anchor for {name} no longer in the oracle source"
    path = tmp_path / f"m_{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"m_{name}.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c99", str(path), "-o", str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
