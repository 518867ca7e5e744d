"""Mutation tests for the oracle's pins (CPU only).

Each case plants one plausible mistake (a dropped term, a wrong sign, divisor
or index, a transposed operand) in a copy of the oracle's C source, compiles
the copy into a temporary directory and requires at least one pin to fail on
it.  The real oracle is never modified.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, original text, replacement, which occurrence of the original: 0-based)
MUTANTS = [
    ("fwd_mean_divisor", "sumsq / (double)D", "sumsq / (double)(D + 1)", 0),
    ("vjp_mean_divisor", "sumsq / (double)D", "sumsq / (double)(D + 1)", 1),
    ("fwd_eps_dropped", "double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / sqrt(ms);", 0),
    ("vjp_eps_dropped", "double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / sqrt(ms);", 1),
    ("fwd_eps_outside_root", "double r = 1.0 / sqrt(ms + eps);",
     "double r = 1.0 / (sqrt(ms) + eps);", 0),
    ("fwd_sumsq_abs", "sumsq += h * h;", "sumsq += h * fabs(h);", 0),
    ("fwd_weight_bias_dropped", "out[i * D + j] = h * r * (weight_bias + w[j]);",
     "out[i * D + j] = h * r * w[j];", 0),
    ("fwd_residual_not_in_sumsq", "double h = ri ? xi[j] + ri[j] : xi[j];",
     "double h = xi[j];", 0),
    ("fwd_residual_not_in_output", "double h = ri ? xi[j] + ri[j] : xi[j];",
     "double h = xi[j];", 1),
    ("fwd_new_residual_is_x", "new_residual[i * D + j] = h;",
     "new_residual[i * D + j] = xi[j];", 0),
    ("fwd_out_transposed", "out[i * D + j] = h", "out[j * rows + i] = h", 0),
    ("vjp_second_term_sign", "- r3_over_d * hi[j] * dot", "+ r3_over_d * hi[j] * dot", 0),
    ("vjp_r_cubed_to_squared", "r * r * r / (double)D", "r * r / (double)D", 0),
    ("vjp_gw_missing_r", "gw[j] += gi[j] * hi[j] * r;", "gw[j] += gi[j] * hi[j];", 0),
    ("vjp_gw_uses_row0", "gw[j] += gi[j] * hi[j] * r;", "gw[j] += gi[j] * x[j] * r;", 0),
    ("vjp_gw_not_zeroed", "gw[j] = 0.0;", "gw[j] = 1.0;", 0),
    ("vjp_dot_without_weight", "dot += gi[j] * (weight_bias + w[j]) * hi[j];",
     "dot += gi[j] * hi[j];", 0),
    ("vjp_dot_g_for_h", "dot += gi[j] * (weight_bias + w[j]) * hi[j];",
     "dot += gi[j] * (weight_bias + w[j]) * gi[j];", 0),
    ("vjp_gx_weight_bias_dropped", "gx[i * D + j] = r * gi[j] * (weight_bias + w[j])",
     "gx[i * D + j] = r * gi[j] * w[j]", 0),
    ("vjp_g_row0", "const double *gi = g + i * D;", "const double *gi = g;", 0),
    ("fused_g_residual_dropped", "g_h[i] = g_h[i] + g_residual[i];", "g_h[i] = g_h[i];", 0),
    ("fused_g_residual_sign", "g_h[i] = g_h[i] + g_residual[i];", "g_h[i] = g_h[i] - g_residual[i];", 0),
    ("silu_exp_sign", "a[j] / (1.0 + exp(-a[j]))", "a[j] / (1.0 + exp(a[j]))", 0),
    ("silu_halves_swapped", "out[i * d + j] = silu * b[j];", "out[i * d + j] = b[j] / (1.0 + exp(-b[j])) * a[j];", 0),
    ("silu_no_gate", "out[i * d + j] = silu * b[j];", "out[i * d + j] = silu;", 0),
    ("silu_row_stride", "const double *a = x + i * 2 * d;", "const double *a = x + i * d;", 0),
    ("silu_second_half_offset", "const double *b = a + d;", "const double *b = a + d - 1;", 0),
    ("rope_sin_sign", "y[ia] = xa * c - xb * s;", "y[ia] = xa * c + xb * s;", 0),
    ("rope_second_sign", "y[ib] = xb * c + xa * s;", "y[ib] = xb * c - xa * s;", 0),
    ("rope_exponent", "pow(base, -2.0 * (double)i / (double)Dh)", "pow(base, -1.0 * (double)i / (double)Dh)", 0),
    ("rope_half_offset", "int64_t ib = interleaved ? 2 * i + 1 : i + Dh / 2;",
     "int64_t ib = interleaved ? 2 * i + 1 : Dh - 1 - i;", 0),
    ("rope_table_swapped", "*c = cos_sin[p * Dh + i];", "*c = cos_sin[p * Dh + Dh / 2 + i];", 0),
    ("rope_token_for_position", "int64_t p = positions[t];", "int64_t p = t;", 0),
    ("kv_v_rotated", "v_cache[(slot * Hkv + h) * Dh + j] = v[(t * Hkv + h) * Dh + j];",
     "v_cache[(slot * Hkv + h) * Dh + j] = k_cache[(slot * Hkv + h) * Dh + j];", 0),
    ("rstd_eps_dropped", "rstd[i] = 1.0 / sqrt(sq / (double)D + eps);",
     "rstd[i] = 1.0 / sqrt(sq / (double)D);", 0),
    ("rstd_residual_ignored", "double hv = residual ? x[i * D + j] + residual[i * D + j] : x[i * D + j];",
     "double hv = x[i * D + j];", 0),
    ("vjp_rstd_row0_scale", "const double rho = rstd[i];", "const double rho = rstd[0];", 0),
    ("vjp_rstd_rho_squared", "rho * rho * rho / (double)D", "rho * rho / (double)D", 0),
    ("vjp_rstd_gw_missing_rho", "gw[j] += g[i * D + j] * x[i * D + j] * rho;",
     "gw[j] += g[i * D + j] * x[i * D + j];", 0),
    ("vjp_rstd_dot_without_weight", "dg += g[i * D + j] * (weight_bias + w[j]) * x[i * D + j];",
     "dg += g[i * D + j] * x[i * D + j];", 0),
    ("vjp_rstd_gx_sign", "- k3 * x[i * D + j] * dg;", "+ k3 * x[i * D + j] * dg;", 0),
    ("kv_slot_is_token", "int64_t slot = slots[t];", "int64_t slot = slots[t] < 0 ? -1 : t % 4;", 0),
]


def _replace_nth(text, old, new, n):
    """Replace the n-th occurrence of ``old``; every target is a C statement,
    so the count is checked against the whole source."""
    assert text.count(old) > n, "mutation target %r has fewer than %d occurrences" % (old, n + 1)
    start = -1
    for _ in range(n + 1):
        start = text.find(old, start + 1)
        assert start >= 0, "mutation target %r (occurrence %d) not in the oracle source" % (old, n)
    return text[:start] + new + text[start + len(old):]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, source, name, old, new, nth):
    mutated = _replace_nth(source, old, new, nth)
    assert mutated != source
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(mutated)
    lib = oracle.compile_source(str(src), str(tmp_path / ("libmutant_%s.so" % name)))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ZeroDivisionError):
            caught.append(pin.__name__)
    assert caught, "no pin catches mutant %s" % name


def test_real_oracle_passes_every_pin():
    orc = oracle.load()
    for pin in ALL_PINS:
        pin(orc)
    assert os.path.exists(oracle.LIB_PATH)
