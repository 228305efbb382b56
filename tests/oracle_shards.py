"""Row-sharded oracle comparisons for workloads too large for one host core.

Batch rows are independent sequences, so the oracle can run on disjoint row ranges in
separate processes: each shard compares every per-row output (H, the cached activations,
d_pre, du, dh0) of its rows with the GPU's, element by element, and returns its own fp64
partial sums of dW and db over its rows.  The caller adds the partials in shard order; that is
the full-batch oracle dW / db up to fp64 rounding (the batch-sum pin of the oracle checks this
decomposition).

Processes are started with the ``spawn`` method, so no worker inherits a CUDA context.
"""
from __future__ import annotations

import concurrent.futures
import multiprocessing
import os

import numpy as np

ROW_KEYS = ("H", "cache", "d_pre", "du", "dh0")
ROW_AXIS = {"H": 1, "cache": 1, "d_pre": 1, "du": 1, "dh0": 0}
IN_ROW_AXIS = {"u": 1, "ts": 1, "dH": 1, "h0": 0}


def _rows(a: np.ndarray, axis: int, r0: int, r1: int) -> np.ndarray:
    return np.ascontiguousarray(a[r0:r1] if axis == 0 else a[:, r0:r1])


def _stats(x: np.ndarray, y: np.ndarray, floor: float) -> dict:
    """max|x - y|, max|y| and max_i |x_i - y_i| / max(|y_i|, floor) of one tensor."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    d = np.abs(x - y)
    ay = np.abs(y)
    return {"max_diff": float(d.max(initial=0.0)), "max_ref": float(ay.max(initial=0.0)),
            "max_elem": float((d / np.maximum(ay, floor)).max(initial=0.0)),
            "finite": bool(np.all(np.isfinite(x)))}


def shard_compare(inp_rows: dict, gpu_rows: dict, floors: dict):
    """One shard: oracle on these rows, stats against the GPU rows, dW / db partials."""
    import oracle

    ref = oracle.step(inp_rows)
    ref["cache"] = np.stack([ref["ff1"], ref["ff2"], ref["gate"]], axis=2)
    stats = {k: _stats(gpu_rows[k], ref[k], floors[k]) for k in gpu_rows}
    return stats, ref["dW"], ref["db"]


def _merge(parts: list[dict]) -> dict:
    out = {}
    for k in parts[0]:
        out[k] = {"max_diff": max(p[k]["max_diff"] for p in parts),
                  "max_ref": max(p[k]["max_ref"] for p in parts),
                  "max_elem": max(p[k]["max_elem"] for p in parts),
                  "finite": all(p[k]["finite"] for p in parts)}
    return out


def compare_all_rows(inp: dict, gpu: dict, n_proc: int | None = None) -> dict:
    """Every row of every per-row output and the full dW / db against the oracle.

    Returns {tensor: {"rel": max|x-y| / max(max|y|, 2^-126), "elem": elementwise relative error
    with a floor of 1e-3 max|y|, "max_ref": max|y|, "finite": ...}}.  The elementwise floor is
    taken from the GPU tensor's own max|x| (known before the shards run; it equals max|y| to
    within the tolerance being checked)."""
    B = inp["h0"].shape[0]
    n_proc = max(1, min(n_proc or os.cpu_count() or 1, B))
    bounds = [(B * i // n_proc, B * (i + 1) // n_proc) for i in range(n_proc)]
    floors = {k: 1e-3 * float(np.max(np.abs(gpu[k]))) for k in ROW_KEYS}
    floors = {k: max(v, 2.0 ** -126) for k, v in floors.items()}
    jobs = []
    for r0, r1 in bounds:
        ir = {k: (_rows(v, IN_ROW_AXIS[k], r0, r1) if k in IN_ROW_AXIS else v)
              for k, v in inp.items()}
        gr = {k: _rows(gpu[k], ROW_AXIS[k], r0, r1) for k in ROW_KEYS}
        jobs.append((ir, gr))
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(max_workers=n_proc, mp_context=ctx) as ex:
        futs = [ex.submit(shard_compare, ir, gr, floors) for ir, gr in jobs]
        res = [f.result() for f in futs]
    stats = _merge([r[0] for r in res])
    dW = np.zeros_like(res[0][1])
    db = np.zeros_like(res[0][2])
    for _, pw, pb in res:  # shard (row) order: a fixed summation order
        dW += pw
        db += pb
    for k, ref in (("dW", dW), ("db", db)):
        floor = max(1e-3 * float(np.max(np.abs(ref))), 2.0 ** -126)
        stats[k] = _stats(gpu[k], ref, floor)
    out = {}
    for k, s in stats.items():
        den = max(s["max_ref"], 2.0 ** -126)
        out[k] = {"rel": s["max_diff"] / den, "elem": s["max_elem"], "max_ref": s["max_ref"],
                  "finite": s["finite"]}
    return out
