"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

Every mutant is a one-token edit of the oracle's C source (a dropped term, a flipped sign, a
wrong index or operand) compiled into a temporary library; the real oracle is never touched.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "cfc_oracle.c")

MUTANTS = {
    "dP_ff1 drops (1 - gate)": ("dp[0 * C + i] = dh * (1.0 - gt) * (1.0 - f1 * f1);",
                                "dp[0 * C + i] = dh * (1.0 - f1 * f1);"),
    "ds sign flipped": ("const double ds = dh * (f2 - f1) * gt * (1.0 - gt);",
                        "const double ds = dh * (f1 - f2) * gt * (1.0 - gt);"),
    "ts scales tb instead of ta": ("sigmoid(P[2] * ts[(size_t)t * B + b] + P[3])",
                                   "sigmoid(P[2] + P[3] * ts[(size_t)t * B + b])"),
    "dP_ta misses ts": ("dp[2 * C + i] = ds * tsv;", "dp[2 * C + i] = ds;"),
    "gate mixes the branches the other way": ("H[o] = f1 * (1.0 - gt) + gt * f2;",
                                              "H[o] = f1 * gt + (1.0 - gt) * f2;"),
    "delta reads the input columns": ("delta[(size_t)b * C + j] = dz[n_x + j];",
                                      "delta[(size_t)b * C + j] = dz[j];"),
    "du reads a shifted column": ("du[row * n_x + k] = dz[k];", "du[row * n_x + k] = dz[k + 1];"),
    "db weighted by z[0]": ("db[m] += a;", "db[m] += a * z[0];"),
    "ff2 uses sigmoid": ("const double f2 = tanh(P[1]);", "const double f2 = sigmoid(P[1]);"),
    "z takes h_t instead of h_{t-1} in dW": (
        "gather_z(B, C, n_x, t, b, u, h0, H, z);\n            const double* dp",
        "gather_z(B, C, n_x, t + 1 < K ? t + 1 : t, b, u, h0, H, z);\n            const double* dp"),
    "W_h transposed in the backward": (
        "acc += W[((size_t)g * C + i) * n_in + k] * dp[g * C + i];",
        "acc += W[((size_t)g * C + (k < n_x ? i : k - n_x)) * n_in + (k < n_x ? k : n_x + i)]"
        " * dp[g * C + i];"),
    "reduce skips the first row": ("for (int r = 0; r < n_batch; ++r)",
                                   "for (int r = 1; r < n_batch; ++r)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin_name, pin in oracle_pins.ALL_PINS.items():
        ok, _ = pin(lib)
        if not ok:
            failed.append(pin_name)
    assert failed, f"no pin caught mutant {name!r}"
