"""Plant plausible mistakes in copies of the tau-decay oracle and check that its pins catch each.

Every mutant is a one-token edit of ``oracle/decay_oracle.c`` compiled into a temporary
library; the real oracle is never touched.  A pin catches a mutant when it fails on it.
"""
import os

import pytest

import oracle
import oracle.decay as decay
import test_oracle_decay_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "decay_oracle.c")

MUTANTS = {
    "decay exponent multiplies by tau": ("const double d = exp(-dt / tau[i]);\n        eo[i]",
                                         "const double d = exp(-dt * tau[i]);\n        eo[i]"),
    "state and candidate swap roles": ("ho[i] = d * hp[i] + (1.0 - d) * e;",
                                       "ho[i] = (1.0 - d) * hp[i] + d * e;"),
    "da drops (1 - d)": ("dat[i] = G[i] * (1.0 - d) * (1.0 - et[i] * et[i]);",
                         "dat[i] = G[i] * (1.0 - et[i] * et[i]);"),
    "dtau sign flipped": ("dtau[i] += G[i] * (hp[i] - et[i]) * d * dt / (tau[i] * tau[i]);",
                          "dtau[i] += G[i] * (et[i] - hp[i]) * d * dt / (tau[i] * tau[i]);"),
    "dtau misses ts": ("dtau[i] += G[i] * (hp[i] - et[i]) * d * dt / (tau[i] * tau[i]);",
                       "dtau[i] += G[i] * (hp[i] - et[i]) * d / (tau[i] * tau[i]);"),
    "carried gradient misses the decay": ("G[i] = G[i] * exp(-dt / tau[i]) + dz[n_x + i];",
                                          "G[i] = G[i] + dz[n_x + i];"),
    "carried gradient reads the input columns": ("G[i] = G[i] * exp(-dt / tau[i]) + dz[n_x + i];",
                                                 "G[i] = G[i] * exp(-dt / tau[i]) + dz[i];"),
    "dW uses h_t instead of h_{t-1}": (
        "decay_gather_z(B, C, n_x, t, b, x, h0, H, z);\n      const double* hp = z + n_x;\n      const double dt = ts[(size_t)t * B + b];\n      const double* dHt",
        "decay_gather_z(B, C, n_x, t + 1 < K ? t + 1 : t, b, x, h0, H, z);\n      const double* hp = z + n_x;\n      const double dt = ts[(size_t)t * B + b];\n      const double* dHt"),
    "db weighted by z[0]": ("db[i] += dat[i];", "db[i] += dat[i] * z[0];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = decay.DecayOracle(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in (pins.test_finite_differences, pins.test_tau_to_zero_is_a_tanh_rnn,
                pins.test_no_time_step_keeps_the_state, pins.test_pure_decay_closed_form,
                pins.test_batch_gradient_is_the_sum_of_rows):
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name!r}"
