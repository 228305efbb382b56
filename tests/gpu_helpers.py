"""Shared helpers of the GPU tests: run the CUDA path through the C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle

H_TOL = 1e-5      # max|x - y| / max|y| on H (and the cached activations)
GRAD_TOL = 1e-4   # same metric on dW, db, du, dh0 (and d_pre)


def run_gpu(inp: dict, dw_mode: int = 0, with_du: bool = True, graph: bool = False) -> dict:
    import torch

    from recurrent_cfc_cell_gb300 import build
    from recurrent_cfc_cell_gb300.step import KLoopStep, to_device

    build.build()
    d = to_device(inp)
    K, B, n_x = inp["u"].shape
    C = inp["h0"].shape[1]
    st = KLoopStep(B, K, C, n_x, dw_mode=dw_mode, with_du=with_du).bind(**d)
    if graph:
        st.capture()
        st.replay()
    else:
        st.run()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in st.outputs().items()}


def oracle_ref(inp: dict) -> dict:
    o = oracle.step(inp)
    o["cache"] = np.stack([o["ff1"], o["ff2"], o["gate"]], axis=2)  # [K,B,3,C]
    return o


def errors(gpu: dict, ref: dict, keys=("H", "cache", "d_pre", "dW", "db", "du", "dh0")) -> dict:
    return {k: oracle.rel_err(gpu[k], ref[k]) for k in keys if k in gpu and k in ref}


def assert_parity(gpu: dict, ref: dict, keys=("H", "cache", "d_pre", "dW", "db", "du", "dh0")):
    errs = errors(gpu, ref, keys)
    for k, e in errs.items():
        tol = H_TOL if k in ("H", "cache") else GRAD_TOL
        assert np.isfinite(e) and e <= tol, f"{k}: rel err {e:.3e} > {tol:g} (all: {errs})"
    return errs
