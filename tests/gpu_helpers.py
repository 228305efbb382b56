"""Shared helpers of the GPU tests: run the CUDA path through the C ABI, compare with the oracle.

Two error measures per tensor, both against the fp64 oracle y:
  rel   max|x - y| / max(max|y|, 2^-126)      -- the gated measure (tolerances below);
  elem  max_i |x_i - y_i| / max(|y_i|, 1e-3 max|y|)  -- elementwise, reported for information.
With CFC_PARITY_REPORT set to a file path, every comparison appends one JSON line there.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

H_TOL = 1e-5      # max|x - y| / max|y| on H (and the cached activations)
GRAD_TOL = 1e-4   # same metric on dW, db, du, dh0 (and d_pre)
KEYS = ("H", "cache", "d_pre", "dW", "db", "du", "dh0")


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (any integer dtype) -> their fp32 values."""
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_rn_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, rounded to nearest, ties to even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def split_planes(d_pre, mp: int, terms: int = 2) -> np.ndarray:
    """fp32 d_pre [K,B,4,C] -> the operand rows a bf16 mode leaves in the workspace head:
    uint16 [K,B,2,mp], hi = bf16(x) and lo = bf16(x - hi); unused entries zero."""
    K, B, _, C = d_pre.shape
    x = np.ascontiguousarray(d_pre, dtype=np.float32).reshape(K, B, 4 * C)
    out = np.zeros((K, B, 2, mp), dtype=np.uint16)
    hi = bf16_rn_bits(x)
    out[:, :, 0, : 4 * C] = hi
    if terms == 2:
        out[:, :, 1, : 4 * C] = bf16_rn_bits(x - bf16_to_f32(hi))
    return out


def decode_dpre(raw, C: int, dw_mode: int) -> np.ndarray:
    """The workspace head after a backward pass -> fp32-valued d_pre [K,B,4,C] (hi + lo for the
    two-term mode, hi alone for the single bf16 term, as is for the fp32 modes)."""
    from recurrent_cfc_cell_gb300 import _lib

    raw = np.asarray(raw)
    if dw_mode in (_lib.CFC_DW_TF32, _lib.CFC_DW_SIMT_FP32):
        return raw
    K, B = raw.shape[:2]
    hi = bf16_to_f32(raw[:, :, 0, : 4 * C]).astype(np.float64)
    if dw_mode == _lib.CFC_DW_ACCURATE:
        hi = hi + bf16_to_f32(raw[:, :, 1, : 4 * C])
    return hi.reshape(K, B, 4, C)


def outputs_np(st) -> dict:
    """A step's outputs as numpy arrays, d_pre decoded to fp32 values."""
    out = {k: v.cpu().numpy() for k, v in st.outputs().items()}
    out["d_pre"] = decode_dpre(out["d_pre"], st.C, st.dw_mode)
    return out


def run_gpu(inp: dict, dw_mode: int = 0, with_du: bool = True, graph: bool = False) -> dict:
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build
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
    # A kernel that abandoned a wait leaves its outputs incomplete; such a run is never compared.
    assert _lib.device_status() == 0, "a kernel reported an abandoned wait"
    return outputs_np(st)


def oracle_ref(inp: dict) -> dict:
    o = oracle.step(inp)
    o["cache"] = np.stack([o["ff1"], o["ff2"], o["gate"]], axis=2)  # [K,B,3,C]
    return o


def elem_err(x, y) -> float:
    """max_i |x_i - y_i| / max(|y_i|, 1e-3 max|y|): the elementwise relative error, with a floor
    where the exact value crosses zero."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if y.size == 0:
        return 0.0
    ay = np.abs(y)
    floor = max(1e-3 * float(ay.max()), oracle.FP32_NORMAL_MIN)
    return float(np.max(np.abs(x - y) / np.maximum(ay, floor)))


def errors(gpu: dict, ref: dict, keys=KEYS) -> dict:
    return {k: oracle.rel_err(gpu[k], ref[k]) for k in keys if k in gpu and k in ref}


def report(case: str, rel: dict, elem: dict | None = None, **extra) -> None:
    """Append one line of measured errors to $CFC_PARITY_REPORT (if set)."""
    path = os.environ.get("CFC_PARITY_REPORT")
    if not path:
        return
    line = {"case": case, "rel": rel, "elem": elem or {}, **extra}
    with open(path, "a") as fh:
        fh.write(json.dumps(line) + "\n")


def tol_for(k: str) -> float:
    return H_TOL if k in ("H", "cache") else GRAD_TOL


def assert_parity(gpu: dict, ref: dict, keys=KEYS, case: str | None = None):
    errs = errors(gpu, ref, keys)
    elem = {k: elem_err(gpu[k], ref[k]) for k in errs}
    if case is None:
        case = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    report(case, errs, elem)
    for k, e in errs.items():
        tol = tol_for(k)
        assert np.isfinite(e) and e <= tol, f"{k}: rel err {e:.3e} > {tol:g} (all: {errs})"
    return errs
