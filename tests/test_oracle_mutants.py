"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is compiled from a textual edit of ``oracle/rope_oracle.c`` into a
temporary folder, on the CPU, and the full pin list is run against it in a
child process (a mutant that crashes counts as caught).  The real oracle is
never modified.
"""
import json
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, [(old, new), ...]) -- each a mistake a hand-written RoPE could contain
MUTANTS = [
    ("y1_sign", [("y[i1] = x1 * c - x2 * s;", "y[i1] = x1 * c + x2 * s;")]),
    ("y2_sign", [("y[i2] = x1 * s + x2 * c;", "y[i2] = -x1 * s + x2 * c;")]),
    ("y1_dropped_term", [("y[i1] = x1 * c - x2 * s;", "y[i1] = x1 * c;")]),
    ("y2_swapped_operands", [("y[i2] = x1 * s + x2 * c;", "y[i2] = x2 * s + x1 * c;")]),
    ("split_half_partner", [("2 * i + 1 : i + h;", "2 * i + 1 : rotary_dim - 1 - i;")]),
    ("interleaved_index", [("? 2 * i : i;", "? 2 * i + 1 : i;"),
                           ("? 2 * i + 1 : i + h;", "? 2 * i : i + h;")]),
    ("frequency_exponent_over_half", [("-(2.0 * (double)i) / (double)rotary_dim",
                                       "-(2.0 * (double)i) / (double)(rotary_dim / 2)")]),
    ("frequency_exponent_sign", [("pow(theta, -(2.0 * (double)i)", "pow(theta, (2.0 * (double)i)")]),
    ("interpolate_multiplies", [("((double)m / interpolate_factor)", "((double)m * interpolate_factor)")]),
    ("backward_ignored", [("double s = backward ? -s_row[i] : s_row[i];", "double s = s_row[i];")]),
    ("cos_sin_swapped", [("cos_out[m * h + i] = cos(a);", "cos_out[m * h + i] = sin(a);"),
                         ("sin_out[m * h + i] = sin(a);", "sin_out[m * h + i] = cos(a);")]),
    ("f32_table_double_rounded_via_bf16",
     [("cos_out[m * h + i] = oracle_f64_to_f32(cos(a));",
       "cos_out[m * h + i] = oracle_f64_to_f32(oracle_bf16_to_f64(oracle_f64_to_bf16(cos(a))));")]),
    ("bf16_truncates", [("n = nearbyint(a / q);", "n = floor(a / q);")]),
    ("rne_ties_away", [("n = nearbyint(a / q);", "n = round(a / q);")]),
    ("f16_bias", [("((E + 15) << 10)", "((E + 14) << 10)")]),
    ("f16_decode_exponent", [("ldexp((double)(1024 + frac), e - 25)", "ldexp((double)(1024 + frac), e - 24)")]),
    ("f16_subnormal_scale", [("ldexp((double)frac, -24)", "ldexp((double)frac, -23)")]),
    ("overflow_not_detected", [("if (v > maxfin)\n        return INFINITY;", "")]),
    ("bf16_decode_shift", [("(uint32_t)bits << 16", "(uint32_t)bits << 15")]),
    ("seq_first_row_as_head_first", [("((b * S + s) * H + hh) * D\n", "((b * H + hh) * S + s) * D\n")]),
    ("gather_ignored", [("cos_tab + r * h, sin_tab + r * h", "cos_tab + s * h, sin_tab + s * h")]),
    ("mask_not_recognised", [("int unrotated = (r == -1);", "int unrotated = 0;")]),
    ("range_check_off_by_one", [("r >= table_rows", "r > table_rows")]),
    ("tail_rerounded", [("else            /* tail: bits copied, never re-rounded */\n"
                         "                            memcpy((char *)y_bits + (row + d) * es,\n"
                         "                                   (const char *)x_in + (row + d) * es, es);",
                         "else store_elem(y_bits, dtype, row + d, 0.0);")]),
    ("tail_dropped_f64", [("for (d = rotary_dim; d < D; ++d)\n        y[d] = x[d];", "")]),
    # frequency modes, row positions, XPOS
    ("pixel_without_pi", [("return M_PI * (1.0 + (double)i", "return (1.0 + (double)i")]),
    ("pixel_spacing_over_h", [("/ (double)(h - 1));", "/ (double)h);")]),
    ("pixel_max_freq_not_halved", [("(max_freq / 2.0 - 1.0)", "(max_freq - 1.0)")]),
    ("constant_mode_uses_theta", [("if (mode == ORACLE_FREQ_CONSTANT)\n        return 1.0;",
                                   "if (mode == ORACLE_FREQ_CONSTANT)\n        return theta;")]),
    ("position_multiplies_divisor", [("return pos_offset + (double)m / pos_divisor;",
                                      "return pos_offset + (double)m * pos_divisor;")]),
    ("position_offset_ignored", [("return pos_offset + (double)m / pos_divisor;",
                                  "return (double)m / pos_divisor;")]),
    ("xpos_zeta_denominator", [("+ gamma) / (1.0 + gamma);", "+ gamma) / (2.0 + gamma);")]),
    ("xpos_zeta_over_half_dim", [("(2.0 * (double)i / (double)rotary_dim + gamma)",
                                  "((double)i / (double)rotary_dim + gamma)")]),
    ("xpos_sign_ignored", [("pow(zeta, (double)sign * (p - center) / base)", "pow(zeta, (p - center) / base)")]),
    ("xpos_centre_ignored", [("pow(zeta, (double)sign * (p - center) / base)", "pow(zeta, (double)sign * p / base)")]),
    ("xpos_base_multiplies", [("pow(zeta, (double)sign * (p - center) / base)",
                               "pow(zeta, (double)sign * (p - center) * base)")]),
    ("xpos_sine_unscaled_f64", [("sin_out[m * h + i] = sc * sin(a);", "sin_out[m * h + i] = sin(a);")]),
    ("xpos_f32_unscaled", [("cos_out[m * h + i] = oracle_f64_to_f32(sc * cos(a));",
                            "cos_out[m * h + i] = oracle_f64_to_f32(cos(a));")]),
]

RUNNER = r"""
import json, sys, traceback
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, oracle_pins
o = oracle.Oracle({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(o)
    except ImportError:
        pass
    except Exception:
        failed.append(pin.__name__)
print(json.dumps(failed))
"""


def _run_mutant(name, edits):
    import oracle

    work = tempfile.mkdtemp(prefix="mutant_%s_" % name)
    o = oracle.load_mutant(edits, work)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=o.path)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if p.returncode != 0:
        return name, ["<crashed rc=%d>" % p.returncode]
    return name, json.loads(p.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def mutant_results():
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        return dict(ex.map(lambda m: _run_mutant(*m), MUTANTS))


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(name, mutant_results):
    caught = mutant_results[name]
    assert caught, "no pin catches the planted mistake %r" % name
