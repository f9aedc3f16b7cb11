"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of the oracle source with one planted mistake (a
dropped term, a wrong sign, a wrong index) and runs the pin tests against
that copy; at least one pin has to fail.  Mistakes are planted on the CPU
only, in a temporary copy; the real oracle is untouched.
"""
import os

import numpy as np
import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = {
    "no_decay": ("double alpha = exp(g * A[i]);", "double alpha = 1.0;"),
    "decay_sign": ("double alpha = exp(g * A[i]);", "double alpha = exp(-g * A[i]);"),
    "erase_sign": ("u = beta * (vvec[j] - r);", "u = beta * (vvec[j] + r);"),
    "no_beta": ("u = beta * (vvec[j] - r);", "u = (vvec[j] - r);"),
    "erase_before_decay": ("for (int i = 0; i < dk; i++) r += S[i * dv + j] * bvec[i];",
                           "for (int i = 0; i < dk; i++) r += S[i * dv + j] * bvec[i] / exp(g * A[i]);"),
    "bwd_dAlog_sign": ("dA_log_unit[(size_t)u * dk + i] = dA[i] * A[i];",
                       "dA_log_unit[(size_t)u * dk + i] = -dA[i] * A[i];"),
    "bwd_dg_drop_A": ("dgt += q * A[i];", "dgt += q;"),
    "bwd_db_drop_erase": ("db_out[at_btHd(b, t, h, i, T, H, dk)] += acc;", "(void)acc;"),
    "bwd_dv_drop_beta": ("dv_out[at_btHd(b, t, h, j, T, H, dv)] = bt * du[j];",
                         "dv_out[at_btHd(b, t, h, j, T, H, dv)] = du[j];"),
    "bwd_no_decay_of_dh": ("for (int j = 0; j < dv; j++) dS[i * dv + j] *= alpha;", ""),
    "chunk_off_by_one": ("for (int s = 0; s <= t; s++) acc += P[t * C + s] * U[s * dv + j];",
                         "for (int s = 0; s < t; s++) acc += P[t * C + s] * U[s * dv + j];"),
}

PIN_CALLS = [
    ("gated_bruteforce", lambda: pins.test_gated_bruteforce_quadratic_form()),
    ("gated_g0", lambda: pins.test_gated_g_zero_is_cumulative_linear_attention()),
    ("worked_example", lambda: pins.test_gated_scalar_worked_example()),
    ("delta_matrix", lambda: pins.test_delta_matrix_product_form()),
    ("delta_replace", lambda: pins.test_delta_replace_invariant()),
    ("delta_beta0", lambda: pins.test_delta_beta_zero_is_pure_decay()),
    ("chunked_gated", lambda: pins.test_chunked_equals_serial("gated", 100, 16)),
    ("chunked_delta", lambda: pins.test_chunked_equals_serial("delta", 100, 16)),
    ("fd_gated", lambda: pins.test_backward_finite_differences("gated", 5, 3)),
    ("fd_delta", lambda: pins.test_backward_finite_differences("delta", 5, 3)),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    monkeypatch.setattr(pins, "oracle", lib)
    caught = []
    for pin, call in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin)
    assert caught, f"no pin caught the planted mistake {name}"


# the chunked reverse mode (numpy) against the serial backward: each planted mistake must break the equality
CHUNKED_SRC = os.path.join(os.path.dirname(oracle.__file__), "chunked_bwd.py")

CHUNKED_MUTANTS = {
    "no_state_decay_grad": ("    dGam[-1] += (dSn * S).sum(axis=1) * E[-1]\n", ""),
    "bh_decay_sign": ('    dGam -= dBh * f["Bh"]\n', '    dGam += dBh * f["Bh"]\n'),
    "solve_not_transposed": ('np.linalg.solve(f["Mmat"].T, dU)', 'np.linalg.solve(f["Mmat"], dU)'),
    "dbeta_drop_K": (' + (dMm * f["K"]).sum(axis=1)', ''),
    "dg_forward_cumsum": ("np.cumsum(dG[::-1])[::-1]", "np.cumsum(dG)"),
    "dQ_strict_mask": ("dQ = (dO @ U.T) * np.tril(np.ones((L, L)))", "dQ = (dO @ U.T) * np.tril(np.ones((L, L)), -1)"),
}


@pytest.mark.parametrize("name", sorted(CHUNKED_MUTANTS))
def test_chunked_backward_pin_catches_planted_mistake(name, tmp_path, monkeypatch):
    import importlib.util
    old, new = CHUNKED_MUTANTS[name]
    src = open(CHUNKED_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    path = tmp_path / "chunked_mutant.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("chunked_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setattr(pins.oracle, "gdn_bwd_chunked", mod.gdn_bwd_chunked)
    caught = []
    for mode in ("gated", "delta"):
        try:
            pins.test_chunked_backward_equals_serial(mode, 37, 16, 4, 5)
        except AssertionError:
            caught.append(mode)
    assert caught, f"no pin caught the chunked-backward mutant {name}"
