"""Planted mistakes in a copy of the oracle must each fail at least one pin (CPU only).

Each case rewrites one expression of ``oracle/sla_oracle.c`` in a temporary
copy (a dropped term, a wrong sign, a wrong index or a transposed operand),
compiles it, and runs the pin battery of ``oracle_pins`` against it.  The
unmodified oracle passes every pin (test_oracle_pins.py); every mutant must not.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "sla_oracle.c")

MUTANTS = [
    ("spmv_wrong_index", "s += values[k] * x[col_idx[k]];", "s += values[k] * x[i];"),
    ("spmv_dropped_term", "for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) s += values[k]",
     "for (int64_t k = row_ptr[i] + 1; k < row_ptr[i + 1]; ++k) s += values[k]"),
    ("dot_wrong_operand", "for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];",
     "for (int64_t i = 0; i < n; ++i) s += a[i] * a[i];"),
    ("x_update_sign", "x[i] = x[i] + alpha * p[i];", "x[i] = x[i] - alpha * p[i];"),
    ("r_update_operand", "r[i] = r[i] - alpha * q[i];", "r[i] = r[i] - alpha * p[i];"),
    ("alpha_transposed", "double alpha = rho / pq;", "double alpha = pq / rho;"),
    ("beta_transposed", "double beta = rho_new / rho;", "double beta = rho / rho_new;"),
    ("p_update_uses_r", "p[i] = z[i] + beta * p[i];", "p[i] = r[i] + beta * p[i];"),
    ("jacobi_multiplies", "z[i] = (precond == 1) ? r[i] / d[i] : r[i];\n    double rho_new",
     "z[i] = (precond == 1) ? r[i] * d[i] : r[i];\n    double rho_new"),
    ("stop_rule_no_sqrt", "if (sqrt(rr) <= rtol * nb) { status = ORC_OK; goto done; }\n    ORC_PARALLEL_FOR",
     "if (rr <= rtol * nb) { status = ORC_OK; goto done; }\n    ORC_PARALLEL_FOR"),
    ("history_off_by_one", "if (history) history[k + 1] = *rel_res;", "if (history) history[k] = *rel_res;"),
    ("grad_values_transposed", "grad_values[k] = -(lambda[i] * x[col_idx[k]]);",
     "grad_values[k] = -(lambda[col_idx[k]] * x[i]);"),
    ("grad_values_sign", "grad_values[k] = -(lambda[i] * x[col_idx[k]]);",
     "grad_values[k] = (lambda[i] * x[col_idx[k]]);"),
    ("adjoint_wrong_rhs", "orc_cg(n, row_ptr, col_idx, values, g, NULL,", "orc_cg(n, row_ptr, col_idx, values, x, NULL,"),
    ("x0_residual_sign", "r[i] = b[i] - q[i];", "r[i] = b[i] + q[i];"),
    ("breakdown_test_dropped", "if (!(pq > 0.0)) { status = ORC_BREAKDOWN; goto done; }", ""),
    ("spmv_transpose_row_for_column", "y[col_idx[k]] = y[col_idx[k]] + values[k] * x[i];",
     "y[col_idx[k]] = y[col_idx[k]] + values[k] * x[col_idx[k]];"),
    ("spmv_transpose_not_transposed", "y[col_idx[k]] = y[col_idx[k]] + values[k] * x[i];",
     "y[i] = y[i] + values[k] * x[col_idx[k]];"),
    ("matvec_grad_transposed", "grad_values[k] = gy[i] * x[col_idx[k]];", "grad_values[k] = gy[col_idx[k]] * x[i];"),
    ("matvec_grad_sign", "grad_values[k] = gy[i] * x[col_idx[k]];", "grad_values[k] = -(gy[i] * x[col_idx[k]]);"),
    ("eig_grad_sign", "acc = acc + ws * (V[s * n + i] * V[s * n + j]);",
     "acc = acc - ws * (V[s * n + i] * V[s * n + j]);"),
    ("eig_grad_drops_weight", "const double ws = w ? w[s] : 1.0;", "const double ws = 1.0;"),
    ("eig_grad_first_vector_only", "for (int64_t s = 0; s < k; ++s) {\n        const double ws",
     "for (int64_t s = 0; s < (k > 0 ? 1 : 0); ++s) {\n        const double ws"),
    ("eig_grad_row_for_column", "acc = acc + ws * (V[s * n + i] * V[s * n + j]);",
     "acc = acc + ws * (V[s * n + i] * V[s * n + i]);"),
    ("eig_grad_wrong_vector", "acc = acc + ws * (V[s * n + i] * V[s * n + j]);",
     "acc = acc + ws * (V[i] * V[j]);"),
    ("transpose_keeps_column", "tr_col_idx[fill[c]] = (int32_t)i;", "tr_col_idx[fill[c]] = (int32_t)c;"),
    ("bicg_beta_ratio_transposed", "const double beta = (rho / rho_prev) * (alpha / omega);",
     "const double beta = (rho / rho_prev) * (omega / alpha);"),
    ("bicg_direction_sign", "p[i] = r[i] + beta * (p[i] - omega * v[i]);", "p[i] = r[i] + beta * (p[i] + omega * v[i]);"),
    ("bicg_s_sign", "s[i] = r[i] - alpha * v[i];", "s[i] = r[i] + alpha * v[i];"),
    ("bicg_omega_transposed", "omega = ts / tt;", "omega = tt / ts;"),
    ("bicg_x_drops_s", "x[i] = (x[i] + alpha * p[i]) + omega * s[i];", "x[i] = x[i] + alpha * p[i];"),
    ("bicg_adjoint_untransposed", "int st = orc_bicgstab(n, trp, tci, tv, g, NULL,",
     "int st = orc_bicgstab(n, row_ptr, col_idx, values, g, NULL,"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, mut, tmp_path):
    text = open(SRC).read()
    assert text.count(orig) == 1, f"mutation site for {name} not unique"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(orig, mut))
    so = str(tmp_path / f"lib{name}.so")
    oracle.build(force=True, src=str(src), out=so)
    lib = oracle.load(so)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant {name} passed every pin"
