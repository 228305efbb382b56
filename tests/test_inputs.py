"""The seeded input recipe (CPU): shapes, dtypes, distributions and structure of the workloads
that both the CUDA path and the oracle read."""
import math

import numpy as np
import pytest

from recurrent_cfc_cell_gb300 import inputs


def _check_common(w, inp):
    K, B, n_x, C, n_in = w.K, w.B, w.n_x, w.C, w.n_in
    shapes = {"u": (K, B, n_x), "h0": (B, C), "W": (4, C, n_in), "b": (4, C), "ts": (K, B),
              "dH": (K, B, C)}
    for k, shp in shapes.items():
        a = inp[k]
        assert a.shape == shp, k
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"], k
    lim = 1.0 / math.sqrt(n_in)
    assert np.all(np.abs(inp["W"]) <= lim * (1 + 1e-6))
    # U(-lim, lim): mean 0, standard deviation lim / sqrt(3)
    assert abs(float(inp["W"].mean())) < 0.05 * lim
    assert abs(float(inp["W"].std()) - lim / math.sqrt(3)) < 0.05 * lim


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_workload_recipe(idx):
    w = inputs.CONFIGS[idx]
    inp = inputs.make_inputs(w)
    _check_common(w, inp)
    if w.bias_std == 0:
        assert np.all(inp["b"] == 0)
    else:
        assert abs(float(inp["b"].std()) - w.bias_std) < 0.25 * w.bias_std
    if w.h0_std == 0:
        assert np.all(inp["h0"] == 0)
    else:
        assert abs(float(inp["h0"].std()) - w.h0_std) < 0.1 * w.h0_std
    if w.ts_range is None:
        assert np.all(inp["ts"] == 1.0)
    else:
        lo, hi = w.ts_range
        assert float(inp["ts"].min()) >= lo and float(inp["ts"].max()) <= hi
    u = inp["u"]
    n_zero = int(np.count_nonzero(u == 0.0))
    assert n_zero == math.floor(w.u_zero_frac * u.size)
    nz = u[u != 0.0]
    assert abs(float(nz.std()) - 1.0) < 0.05
    assert np.all(inp["dH"] != 0.0)  # an upstream gradient at every step


def test_stress_recipe_structure_on_a_smaller_batch():
    """The stress workload's ts range and last-8-steps upstream gradient, at B = 16."""
    s = inputs.CONFIGS[4]
    w = inputs.custom(B=16, K=s.K, n_x=s.n_x, C=s.C, seed=s.seed, ts_range=s.ts_range,
                      dH_last=s.dH_last)
    inp = inputs.make_inputs(w)
    _check_common(w, inp)
    dH = inp["dH"]
    assert np.all(dH[: w.K - 8] == 0.0)
    assert np.all(dH[w.K - 8:] != 0.0)
    assert float(inp["ts"].min()) >= 0.1 and float(inp["ts"].max()) <= 4.0


def test_same_seed_same_arrays_other_seed_other_arrays():
    w = inputs.custom(B=3, K=4, n_x=5, C=6, seed=11)
    a, b = inputs.make_inputs(w), inputs.make_inputs(w)
    c = inputs.make_inputs(inputs.custom(B=3, K=4, n_x=5, C=6, seed=12))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    assert not np.array_equal(a["W"], c["W"])
