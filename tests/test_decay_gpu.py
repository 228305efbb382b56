"""The pages' tau-decay cell on the GPU (cfc_decay_forward / cfc_decay_backward) against its fp64
oracle, element by element, with the four-gate cell's tolerances: 1e-5 on H and E = tanh(a),
1e-4 on dW, db, dtau, dx and dh0 (max|x - y| / max|y| per tensor)."""
import numpy as np
import pytest

import oracle
import oracle.decay as decay
from recurrent_cfc_cell_gb300 import inputs

from gpu_helpers import elem_err, report

pytestmark = pytest.mark.gpu

H_TOL, GRAD_TOL = 1e-5, 1e-4
OUTS = ("H", "E", "dW", "db", "dtau", "dx", "dh0")

# The three workloads (tiny; the pages' shape, 128 inputs and 128 hidden units; a larger
# batch), and ragged ones: odd sizes, C below 32 / 64 / 128, batches that take 1, 2 and 4 rows
# per CTA, and one- and two-step sequences (the BPTT's input ring barely filled).
SHAPES = [(w.B, w.K, w.n_x, w.C, w.seed) for w in inputs.DECAY_CONFIGS] + [
    (7, 11, 13, 100, 21), (5, 6, 3, 17, 22), (9, 5, 40, 64, 23), (300, 4, 24, 128, 24),
    (700, 3, 16, 96, 25), (9, 1, 8, 64, 26), (6, 2, 5, 33, 27)]


def _ids(s):
    return "B{}_K{}_nx{}_C{}".format(*s[:4])


def run_decay(inp: dict, with_dx: bool = True) -> dict:
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    d = {k: torch.from_numpy(v).cuda().contiguous() for k, v in inp.items()}
    K, B, n_x = inp["x"].shape
    C = inp["h0"].shape[1]
    dev = d["x"].device
    f = dict(dtype=torch.float32, device=dev)
    H = torch.full((K, B, C), float("nan"), **f)
    E = torch.full((K, B, C), float("nan"), **f)
    _lib.cfc_decay_forward(d["x"], d["h0"], d["W"], d["b"], d["tau"], d["ts"], H, E)
    out = {k: torch.full(v, float("nan"), **f) for k, v in
           (("dW", (C, n_x + C)), ("db", (C,)), ("dtau", (C,)), ("dh0", (B, C)))}
    out["dx"] = torch.full((K, B, n_x), float("nan"), **f) if with_dx else None
    ws = torch.empty(_lib.decay_workspace_bytes(B, K, C, n_x), dtype=torch.uint8, device=dev)
    _lib.cfc_decay_backward(d["dH"], d["x"], d["h0"], d["W"], d["tau"], d["ts"], H, E,
                            out["dW"], out["db"], out["dtau"], out["dx"], out["dh0"], ws)
    torch.cuda.synchronize()
    assert _lib.device_status() == 0
    got = {"H": H.cpu().numpy(), "E": E.cpu().numpy()}
    got.update({k: v.cpu().numpy() for k, v in out.items() if v is not None})
    return got


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
def test_decay_matches_oracle(shape):
    B, K, n_x, C, seed = shape
    inp = inputs.make_decay_inputs(inputs.decay_custom(B, K, n_x, C, seed=seed))
    got = run_decay(inp)
    ref = decay.step(inp)
    rel = {k: oracle.rel_err(got[k], ref[k]) for k in OUTS}
    report("decay::" + _ids(shape), rel, {k: elem_err(got[k], ref[k]) for k in OUTS})
    for k in OUTS:
        tol = H_TOL if k in ("H", "E") else GRAD_TOL
        assert np.isfinite(rel[k]) and rel[k] <= tol, (k, rel[k], tol)


def test_decay_is_bitwise_reproducible_and_dx_optional():
    inp = inputs.make_decay_inputs(inputs.DECAY_CONFIGS[1])
    a = run_decay(inp)
    b = run_decay(inp)
    for k in OUTS:
        assert np.array_equal(a[k], b[k]), k
    c = run_decay(inp, with_dx=False)
    for k in ("dW", "db", "dtau", "dh0"):
        assert np.array_equal(a[k], c[k]), k
