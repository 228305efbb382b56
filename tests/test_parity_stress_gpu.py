"""The throughput-stress workload (B=2048, K=128, n_x=64, C=256) against the fp64 oracle on
every row, in the launch configuration the benchmark times (cfc_forward_backward).

The oracle runs on all 2048 rows, split by rows over spawned host processes (rows are
independent sequences): H, the cached activations, d_pre, du and dh0 are compared element by
element on every row, and dW / db against the sum of the shards' fp64 partials.  On this
workload the upstream gradient is nonzero only at the last 8 of 128 steps, so the exact dh0 is
about 1e-51, below fp32's normal range, and its check is only absolute; the second case keeps
the same shape with K = 16, where dh0 is well inside fp32's range and the tensor-core BPTT's
dh0 is checked with relative precision."""
import dataclasses

import numpy as np
import pytest

from gpu_helpers import report, run_gpu, tol_for
from oracle_shards import compare_all_rows
from recurrent_cfc_cell_gb300 import inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STRESS = inputs.CONFIGS[4]
STRESS_K16 = dataclasses.replace(STRESS, name="stress_B2048_K16_nx64_C256", K=16)


@pytest.mark.parametrize("w", [STRESS, STRESS_K16], ids=lambda w: w.name)
def test_stress_shape_every_row_against_the_oracle(w):
    inp = inputs.make_inputs(w)
    gpu = run_gpu(inp)
    res = compare_all_rows(inp, gpu)
    report(f"all_rows::{w.name}", {k: v["rel"] for k, v in res.items()},
           {k: v["elem"] for k, v in res.items()},
           max_ref={k: v["max_ref"] for k, v in res.items()})
    for k, v in res.items():
        assert v["finite"], k
        assert v["rel"] <= tol_for(k), (k, v, res)
    if w.K <= 16:
        # dH reaches h0 through at most 16 steps: dh0 must be a normal fp32 magnitude, so the
        # check above is a relative one.
        assert res["dh0"]["max_ref"] > 1e-20, res["dh0"]
    assert np.isfinite(res["dW"]["max_ref"]) and res["dW"]["max_ref"] > 0
