"""The bf16 state variant (cfc_forward_bf16 / cfc_backward_bf16): H, the cache and d_pre stored
as bf16, every sum in fp32.

The forward's recurrence carries h in fp32 exactly as cfc_forward does, so its bf16 H and cache
must be bitwise the fp32 results rounded to nearest even.  The backward reads the rounded cache
and contracts bf16 operands, so it is compared with the fp64 oracle under the tolerance derived
in the design notes (reading R14)."""
import numpy as np
import pytest

from recurrent_cfc_cell_gb300 import inputs

from gpu_helpers import bf16_rn_bits, elem_err, oracle_ref, report

pytestmark = pytest.mark.gpu

# Max-normalised error bounds of the variant against the fp64 oracle (reading R14): H and the
# cache are the fp32 results (within 1e-5 of the oracle) rounded to bf16, a relative error of
# at most 2^-8; every product of the backward takes operands rounded to bf16 (2^-7 per
# product), and the bound allows twice that for the K-step recurrence and the sums.
BF16_H_TOL = 2.0 ** -8 + 1e-5
BF16_GRAD_TOL = 2.0 ** -6

# CUDA-core forward and BPTT (register path), the pages' shape, a ragged odd-n_x shape, a
# shape whose BPTT takes the shared-memory ring (more than 4 rows per cluster), and shapes on
# the tensor-core recurrences (C = 256 from 129 rows for the BPTT, 384 for the forward).
SHAPES = [dict(B=32, K=64, n_x=48, C=128), dict(B=7, K=11, n_x=13, C=100),
          dict(B=500, K=4, n_x=16, C=128), dict(B=200, K=5, n_x=8, C=256),
          dict(B=800, K=4, n_x=16, C=256), dict(B=400, K=3, n_x=80, C=256)]


def _ids(s):
    return "B{B}_K{K}_nx{n_x}_C{C}".format(**s)


def _run(shape, seed):
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build
    from recurrent_cfc_cell_gb300.step import to_device

    build.build()
    inp = inputs.make_inputs(inputs.custom(seed=seed, **shape))
    d = to_device(inp)
    B, K, C, n_x = shape["B"], shape["K"], shape["C"], shape["n_x"]
    dev = d["u"].device
    H16 = torch.empty((K, B, C), dtype=torch.bfloat16, device=dev)
    c16 = torch.empty((K, B, 3, C), dtype=torch.bfloat16, device=dev)
    fws = torch.empty(_lib.forward_bf16_workspace_bytes(B, K, C, n_x), dtype=torch.uint8,
                      device=dev)
    _lib.cfc_forward_bf16(d["u"], d["h0"], d["W"], d["b"], d["ts"], H16, c16, fws)
    out = {k: torch.empty(v, device=dev) for k, v in
           (("dW", (4, C, n_x + C)), ("db", (4, C)), ("du", (K, B, n_x)), ("dh0", (B, C)))}
    ws = torch.empty(_lib.workspace_bytes(B, K, C, n_x, _lib.CFC_DW_BF16), dtype=torch.uint8,
                     device=dev)
    _lib.cfc_backward_bf16(d["dH"], d["u"], d["h0"], d["W"], d["ts"], H16, c16, out["dW"],
                           out["db"], out["du"], out["dh0"], ws)
    torch.cuda.synchronize()
    assert _lib.device_status() == 0
    return inp, d, H16, c16, out


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
def test_forward_bf16_is_the_fp32_forward_rounded(shape):
    import torch

    from recurrent_cfc_cell_gb300 import _lib

    inp, d, H16, c16, _ = _run(shape, seed=41)
    K, B, C = H16.shape
    H = torch.empty((K, B, C), device=H16.device)
    cache = torch.empty((K, B, 3, C), device=H16.device)
    _lib.cfc_forward(d["u"], d["h0"], d["W"], d["b"], d["ts"], H, cache)
    torch.cuda.synchronize()
    got_h = H16.view(torch.int16).cpu().numpy().view(np.uint16)
    got_c = c16.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_h, bf16_rn_bits(H.cpu().numpy()))
    assert np.array_equal(got_c, bf16_rn_bits(cache.cpu().numpy()))


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
def test_bf16_state_matches_oracle(shape):
    import torch

    inp, d, H16, c16, out = _run(shape, seed=43)
    ref = oracle_ref(inp)
    got = {"H": H16.float().cpu().numpy(), "cache": c16.float().cpu().numpy()}
    got.update({k: v.cpu().numpy() for k, v in out.items()})
    rel, elem = {}, {}
    for k, g in got.items():
        y = ref[k]
        rel[k] = float(np.max(np.abs(g.astype(np.float64) - y)) / max(np.max(np.abs(y)), 1e-300))
        elem[k] = elem_err(g, y)
    report("bf16_state::" + _ids(shape), rel, elem)
    for k, e in rel.items():
        tol = BF16_H_TOL if k in ("H", "cache") else BF16_GRAD_TOL
        assert np.isfinite(e) and e <= tol, (k, e, tol)
