"""The fp64 oracle against facts other than itself (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins
from recurrent_cfc_cell_gb300 import inputs


@pytest.fixture(scope="module")
def lib():
    return oracle.default()


@pytest.mark.parametrize("name", sorted(oracle_pins.ALL_PINS))
def test_pin(lib, name):
    ok, detail = oracle_pins.ALL_PINS[name](lib)
    assert ok, f"{name}: {detail}"


def test_finite_difference_tiny_workload(lib):
    """Central differences on every gradient entry of the tiny workload (B=4, K=8, C=32)."""
    inp = {k: np.array(v, dtype=np.float64)
           for k, v in inputs.make_inputs(inputs.CONFIGS[0]).items()}
    # The tiny workload has zero biases and h0; finite differences need no change for that.
    ok, errs = oracle_pins.pin_finite_difference(lib, inp, tol=1e-6)
    assert ok, errs


def test_forward_outputs_bounded(lib):
    """tanh and sigmoid bound every cached activation; h is a convex mix of ff1 and ff2."""
    inp = inputs.make_inputs(inputs.CONFIGS[1])
    o = lib.forward(inp)
    assert np.all(np.abs(o["ff1"]) < 1) and np.all(np.abs(o["ff2"]) < 1)
    assert np.all((o["gate"] > 0) & (o["gate"] < 1))
    lo = np.minimum(o["ff1"], o["ff2"]) - 1e-15
    hi = np.maximum(o["ff1"], o["ff2"]) + 1e-15
    assert np.all((o["H"] >= lo) & (o["H"] <= hi))


def test_stress_upstream_gradient_support(lib):
    """With dH nonzero only at the last 8 steps, d_pre at steps before them comes only from
    the recurrence; at K=12 it is still nonzero at t=0 (the chain reaches back)."""
    w = inputs.custom(B=2, K=12, n_x=3, C=4, seed=3, dH_last=8)
    inp = inputs.make_inputs(w)
    assert np.all(inp["dH"][:4] == 0) and np.all(inp["dH"][4:] != 0)
    o = lib.backward(inp)
    assert np.max(np.abs(o["d_pre"][0])) > 0
