"""Every plausible mistake planted in a copy of the oracle trips a pin.

Each mutant is a textual edit of the oracle's C source, compiled into a
temporary library on the CPU; the real source is never modified. A mutant
that passes every pin would mean the pins cannot tell that mistake apart from
a correct oracle.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rmsnorm_oracle.c")

# (name, text to replace, replacement, which occurrence (0-based) or None = all)
MUTANTS = [
    ("eps_dropped", "sum_sq / (double)N + eps", "sum_sq / (double)N", None),
    ("eps_outside_sqrt", "1.0 / sqrt(sum_sq / (double)N + eps)",
     "1.0 / sqrt(sum_sq / (double)N) + eps", None),
    ("mean_over_padded_width", "sum_sq / (double)N", "sum_sq / (double)(N + 1)", None),
    ("no_square_root", "1.0 / sqrt(", "1.0 / (", None),
    ("sum_not_squared", "sum_sq += v * v;", "sum_sq += v;", None),
    ("fwd_weight_by_row", "load_as_double(w, w_dtype, j);\n    }\n    return ORACLE_OK;",
     "load_as_double(w, w_dtype, i);\n    }\n    return ORACLE_OK;", None),
    ("fwd_weight_dropped", "* r *\n                                   load_as_double(w, w_dtype, j);",
     "* r;", None),
    ("fwd_weight_decoded_as_x", "load_as_double(w, w_dtype, j);\n    }\n    return ORACLE_OK;",
     "load_as_double(w, dtype, j);\n    }\n    return ORACLE_OK;", None),
    ("dx_sign_flipped", "r * (g - xhat * c)", "r * (g + xhat * c)", None),
    ("dx_correction_dropped", "r * (g - xhat * c)", "r * g", None),
    ("dx_outer_r_dropped", "r * (g - xhat * c)", "(g - xhat * c)", None),
    ("dx_mean_not_divided", "c /= (double)N;", "", None),
    ("dx_gain_dropped", "double g = load_as_double(dy, dtype, i * N + j) *\n"
                        "                       load_as_double(w, w_dtype, j);\n"
                        "            dx_out", "double g = load_as_double(dy, dtype, i * N + j);\n"
                                            "            dx_out", None),
    ("dx_x_for_dy", "double g = load_as_double(dy, dtype, i * N + j) *\n"
                    "                       load_as_double(w, w_dtype, j);\n            c +=",
     "double g = load_as_double(x, dtype, i * N + j) *\n"
     "                       load_as_double(w, w_dtype, j);\n            c +=", None),
    ("dx_weight_decoded_as_x", "load_as_double(w, w_dtype, j);\n            dx_out",
     "load_as_double(w, dtype, j);\n            dx_out", None),
    ("dw_extra_r", "dw_out[j] += load_as_double(dy, dtype, i * N + j) * xhat;",
     "dw_out[j] += load_as_double(dy, dtype, i * N + j) * xhat * r;", None),
    ("dw_x_for_dy", "dw_out[j] += load_as_double(dy,", "dw_out[j] += load_as_double(x,", None),
    ("dw_last_row_skipped", "for (i = 0; i < M; ++i) {", "for (i = 0; i + 1 < M; ++i) {", None),
    ("dw_transposed_index", "dw_out[j] += load_as_double(dy, dtype, i * N + j)",
     "dw_out[j] += load_as_double(dy, dtype, j * M + i)", None),
    ("bf16_wrong_shift", "<< 16;", "<< 15;", None),
    ("f16_wrong_bias", "ldexp(1.0 + (double)m / 1024.0, e - 15)",
     "ldexp(1.0 + (double)m / 1024.0, e - 16)", None),
    ("f16_subnormal_scale", "ldexp((double)m, -24)", "ldexp((double)m, -25)", None),
    ("f16_sign_dropped", "return sign ? -v : v;", "return v;", None),
    ("f16_implicit_one_dropped", "ldexp(1.0 + (double)m / 1024.0", "ldexp((double)m / 1024.0", None),
    ("row_selection_ignored", "return rows ? rows[k] : k;", "return k;", None),
    ("add_sum_not_rounded",
     "return round_to_dtype(load_as_double(x, dtype, k) + load_as_double(res, dtype, k), dtype);",
     "return load_as_double(x, dtype, k) + load_as_double(res, dtype, k);", None),
    ("add_residual_dropped",
     "load_as_double(x, dtype, k) + load_as_double(res, dtype, k)",
     "load_as_double(x, dtype, k)", None),
    ("add_y_of_x_not_h", "y_out[k * N + j] = h * r * load_as_double(w, w_dtype, j);",
     "y_out[k * N + j] = load_as_double(x, dtype, i * N + j) * r * load_as_double(w, w_dtype, j);",
     None),
    ("add_sum_sq_of_x", "double h = stored_sum(x, res, dtype, i * N + j);\n            sum_sq += h * h;",
     "double h = load_as_double(x, dtype, i * N + j);\n            sum_sq += h * h;", None),
    ("add_dres_dropped", "dx_out[k * N + j] += load_as_double(dres, dtype, i * N + j);",
     "dx_out[k * N + j] += 0.0;", None),
    ("add_dres_sign", "dx_out[k * N + j] += load_as_double(dres",
     "dx_out[k * N + j] -= load_as_double(dres", None),
    ("add_dres_row_index", "load_as_double(dres, dtype, i * N + j)",
     "load_as_double(dres, dtype, k * N + j)", None),
    ("round_ties_away", "nearbyint(v / q)", "round(v / q)", None),
    ("round_one_bit_short", "e - (p - 1)", "e - (p - 2)", None),
    ("round_no_subnormal_floor", "if (e < emin)\n        e = emin;", "", None),
    ("round_no_overflow", "return copysign(INFINITY, v);", "return r;", None),
    ("round_f16_exponent_range", "round_to_format(v, 11, -14, 15)",
     "round_to_format(v, 11, -15, 15)", None),
    ("round_bf16_precision", "round_to_format(v, 8, -126, 127)",
     "round_to_format(v, 7, -126, 127)", None),
    ("round_bf16_as_f32", "round_to_format(v, 8, -126, 127)",
     "round_to_format(v, 24, -126, 127)", None),
]


def _mutant_source(old, new, which):
    src = open(SRC).read()
    count = src.count(old)
    assert count >= 1, f"mutation anchor not found: {old!r}"
    if which is None:
        return src.replace(old, new)
    parts = src.split(old)
    return old.join(parts[:which + 1]) + new + old.join(parts[which + 1:])


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, which):
    src = tmp_path / f"{name}.c"
    src.write_text(_mutant_source(old, new, which))
    lib_path = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(lib_path),
                    str(src), "-lm"], check=True)
    mutant = oracle.Oracle(oracle.load(str(lib_path)))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError) as e:
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"
