"""Planted-mistake check for the oracle's pins.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign or index, a swapped operand, a wrong tie rule),
builds it with the same flags into a temporary directory and runs every pin
on it. At least one pin must fail, or the pins would not catch that mistake.
The real oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "tko_oracle.c")

MUTANTS = {
    "sigmoid_sign": ("exp(-g)", "exp(g)"),
    "up_reads_gate": ("xr[hidden + i]", "xr[i]"),
    "weight_dropped": ("silu * u * w", "silu * u"),
    "ties_to_odd": ("(c & 1) == 0", "(c & 1) == 1"),
    "ue8m0_clamp_lo": ("if (k < -127)\n        k = -127;", "if (k < -126)\n        k = -126;"),
    "ue8m0_clamp_dropped": ("if (k < -127)\n        k = -127;", ""),
    "fp32_scale_by_reciprocal": ("float s = amax / qmax;", "float s = amax * (1.0f / qmax);"),
    "ue8m0_off_by_one": ("qmax * ldexp(1.0, k) < (double)amax", "qmax * ldexp(1.0, k) <= (double)amax"),
    "scale_inverted": ("float s = amax / qmax;", "float s = qmax / amax;"),
    "up_clamp_one_sided": ("} else if (u < -lim) {", "} else if (u < -2 * lim) {"),
    "gate_clamp_not_strict": ("if (g > lim) {", "if (g >= lim) {"),
    "nibbles_swapped": ("(codes[2 * k] & 0xF) | ((codes[2 * k + 1] & 0xF) << 4)",
                        "(codes[2 * k + 1] & 0xF) | ((codes[2 * k] & 0xF) << 4)"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e2m1_bias": ("ldexp(1.0 + (double)m / 2.0, e - 1)", "ldexp(1.0 + (double)m / 2.0, e - 2)"),
    "group_offset": ("y + r * hidden + j * group", "y + r * hidden + j"),
    "scale_index": ("[r * ngroups + j] = sf", "[j * rows + r] = sf"),
    "amax_min": ("if (a > amax)", "if (a < amax)"),
    "bf16_shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "zero_scale_kept": ("    if (s == 0.0f)\n        s = 1.0f;", ""),
    "quotient_multiplied": ("float quotient = y[i] / s;", "float quotient = y[i] * s;"),
    "packed_byte_order": ("[4 * ((j / 4) * ld + t) + (j % 4)]", "[4 * ((j / 4) * ld + t) + (3 - j % 4)]"),
    "column_major_transposed": ("((float *)out)[j * ld + t] = v;", "((float *)out)[t * ld + j] = v;"),
    "transposed_index_swapped": ("out[i * ld + t] = t < rows ? q[t * hidden + i] : 0;",
                                 "out[i * ld + t] = t < rows ? q[i * rows + t] : 0;"),
    "transposed_padding_kept": ("out[i * ld + t] = t < rows ? q[t * hidden + i] : 0;",
                                "if (t < rows) out[i * ld + t] = q[t * hidden + i];"),
    "backward_dsilu_drops_one_minus_sigmoid": ("dsilu = sig * (1.0 + g * (1.0 - sig));",
                                               "dsilu = sig * (1.0 + g * sig);"),
    "backward_dsilu_sign": ("dsilu = sig * (1.0 + g * (1.0 - sig));", "dsilu = sig * (1.0 - g * (1.0 - sig));"),
    "backward_gate_mask_ignored": ("pass_g ? d * wr * u * dsilu : 0.0", "d * wr * u * dsilu"),
    "backward_up_mask_ignored": ("pass_u ? d * wr * silu : 0.0", "d * wr * silu"),
    "backward_dw_drops_up": ("acc += d * silu * u;", "acc += d * silu;"),
    "backward_weight_dropped": ("pass_g ? d * wr * u * dsilu : 0.0", "pass_g ? d * u * dsilu : 0.0"),
    "cols_gather_transposed": ("col[r] = y[r * hidden + j];", "col[r] = y[j * rows + r];"),
    "cols_store_transposed": ("q[r * hidden + j] = codes[r];", "q[j * rows + r] = codes[r];"),
    "cols_nibbles_swapped": ("if (j % 2 == 0)\n                    *byte", "if (j % 2 == 1)\n                    *byte"),
    "cols_last_row_dropped": ("quantize_group(col, rows, scale_fmt", "quantize_group(col, rows - 1, scale_fmt"),
    "cols_scale_index": ("((float *)scales)[j] = sf;", "((float *)scales)[j / 2] = sf;"),
    "reduce_weight_dropped": ("acc += (double)w[t * K + k] * v;", "acc += v;"),
    "reduce_empty_slot_kept": ("if (r < 0)\n                    continue;", "if (r < 0)\n                    r = 0;"),
    "reduce_global_scale_dropped": ("bf16_rne_from_double((double)gs * acc)", "bf16_rne_from_double(acc)"),
    "reduce_fp8_scale_index": ("y_scale[r * (hidden / 128) + i / 128]", "y_scale[r * (hidden / 128)]"),
    "reduce_bf16_ties_odd": ("pick = ((lo_bits >> 16) & 1) ? hi_bits : lo_bits;", "pick = ((lo_bits >> 16) & 1) ? lo_bits : hi_bits;"),
}


def _run_pins(lib):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, OverflowError, FloatingPointError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, "mutation site not found: %r" % old
    mutated = tmp_path / "mutant.c"
    mutated.write_text(text.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", str(so), str(mutated), "-lm"])
    lib = oracle.load(str(so))
    failed = _run_pins(lib)
    assert failed, "no pin caught the planted mistake %r" % name
