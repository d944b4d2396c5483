"""Plant plausible mistakes in a copy of the oracle and require the pins to
catch every one (CPU only).

Each mutant is a one-place textual edit of the oracle's C source: a dropped
term, a wrong sign, index or bound, a transposed operand.  The copy is
compiled into a temporary shared object and every pin runs against it; the
test passes only if at least one pin fails for each mutant.  All edits keep
memory accesses in bounds, so a mutant can give wrong numbers but not crash.
"""
import os

import pytest

import oracle
import oracle_pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

MUTANTS = {
    "relu_dropped": ("const double r = d > 0.0 ? d : 0.0;", "const double r = d;"),
    "relu_inverted": ("const double r = d > 0.0 ? d : 0.0;", "const double r = d < 0.0 ? d : 0.0;"),
    "scale_dropped": ("total += r * (double)kv_scale * (double)w_row[h];",
                      "total += r * (double)w_row[h];"),
    "weight_dropped": ("total += r * (double)kv_scale * (double)w_row[h];",
                       "total += r * (double)kv_scale;"),
    "weights_reversed": ("total += r * (double)kv_scale * (double)w_row[h];",
                         "total += r * (double)kv_scale * (double)w_row[heads - 1 - h];"),
    "head_sum_overwrites": ("total += r * (double)kv_scale", "total = r * (double)kv_scale"),
    "dot_drops_last_term": ("for (int d = 0; d < dim; ++d)", "for (int d = 0; d < dim - 1; ++d)"),
    "dot_reversed_operand": ("oracle_e4m3_to_double(b[d]);", "oracle_e4m3_to_double(b[dim - 1 - d]);"),
    "q_head_stride": ("dot_e4m3(q_row + (size_t)h * dim, k_row, dim)", "dot_e4m3(q_row, k_row, dim)"),
    "e4m3_bias": ("mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);",
                  "mag = ldexp(1.0 + (double)mant / 8.0, expo - 8);"),
    "e4m3_mantissa": ("mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);",
                      "mag = ldexp(1.0 + (double)mant / 16.0, expo - 7);"),
    "e4m3_subnormal": ("mag = ldexp((double)mant / 8.0, 1 - 7);", "mag = ldexp((double)mant / 8.0, -7);"),
    "e4m3_sign": ("return sign ? -mag : mag;", "return mag;"),
    "e4m3_nan": ("if (expo == 0xF && mant == 0x7) return NAN;", "if (expo == 0xF && mant == 0x7) return 480.0;"),
    "decode_window_exclusive": ("return p >= 0 && p <= last && p < a->max_model_len;",
                                "return p >= 0 && p < last && p < a->max_model_len;"),
    "decode_window_no_next_n": ("(int64_t)a->context_lens[b] - a->next_n + n;",
                                "(int64_t)a->context_lens[b] - 1;"),
    "decode_slot_shift": ("const int64_t slot = p % a->block_size;",
                          "const int64_t slot = (p + 1) % a->block_size;"),
    "decode_table_row": ("a->block_tables[(int64_t)b * a->max_blocks + blk];",
                         "a->block_tables[blk];"),
    "decode_scale_slot": ("+ (int64_t)a->block_size * a->dim + 4 * slot;",
                          "+ (int64_t)a->block_size * a->dim;"),
    "decode_q_row": ("const uint8_t* q_row = a->q + row * a->heads * a->dim;",
                     "const uint8_t* q_row = a->q + (int64_t)b * a->next_n * a->heads * a->dim;"),
    "decode_weight_row": ("const float* w_row = a->weights + row * a->heads;",
                          "const float* w_row = a->weights + (int64_t)n * a->heads;"),
    "prefill_ke_inclusive": ("if (hi > a->cols) hi = a->cols;\n  return n >= lo && n < hi;",
                             "if (hi > a->cols) hi = a->cols;\n  return n >= lo && n <= hi;"),
    "prefill_no_clamp_low": ("if (lo < 0) lo = 0;", "if (lo < 0) lo = 1;"),
    "prefill_weight_row": ("a->weights + m * a->heads,", "a->weights + 0 * m * a->heads,"),
    "prefill_scale_index": ("a->k + n * a->dim, a->kv_scale[n],", "a->k + n * a->dim, a->kv_scale[0],"),
}


def _source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "fp8idx_oracle.c")) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = _source()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libmutant.so")))
    o = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
