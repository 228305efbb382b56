"""fp64 CPU oracle for the CfC K-loop (forward, BPTT, weight gradient, axis-0 reduction).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this package.

The arithmetic lives in ``cfc_oracle.c`` (plain C, fp64, single thread); this module builds it
with gcc and marshals numpy arrays through ctypes.  Inputs are converted to fp64 from whatever
precision the caller holds (normally the fp32 arrays both sides consume).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cfc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libcfc_oracle.so")
_lock = threading.Lock()
_lib = None


GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source to a shared library (atomic replace)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction) and return the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


class OracleLib:
    """ctypes view of one build of the oracle (the default build, or a test's own variant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.cfc_oracle_forward.argtypes = [i, i, i, i] + [dp] * 9
        lib.cfc_oracle_forward.restype = i
        lib.cfc_oracle_backward.argtypes = [i, i, i, i] + [dp] * 14
        lib.cfc_oracle_backward.restype = i
        lib.cfc_oracle_loss.argtypes = [i, i, i, dp, dp]
        lib.cfc_oracle_loss.restype = ctypes.c_double
        lib.cfc_oracle_reduce_axis0.argtypes = [i, i, dp, dp]
        lib.cfc_oracle_reduce_axis0.restype = i
        self.lib = lib
        self.path = path

    def forward(self, inp: dict) -> dict:
        """H [K,B,C] and the cached activations ff1, ff2, gate [K,B,C], all fp64."""
        B, K, C, n_x = _dims(inp)
        u, h0, W, b, ts = (_f64(inp[k]) for k in ("u", "h0", "W", "b", "ts"))
        H = np.empty((K, B, C))
        ff1, ff2, gate = np.empty_like(H), np.empty_like(H), np.empty_like(H)
        rc = self.lib.cfc_oracle_forward(B, K, C, n_x, _p(u), _p(h0), _p(W), _p(b), _p(ts),
                                         _p(H), _p(ff1), _p(ff2), _p(gate))
        if rc != 0:
            raise ValueError(f"cfc_oracle_forward failed: {rc}")
        return {"H": H, "ff1": ff1, "ff2": ff2, "gate": gate}

    def loss(self, inp: dict, fwd: dict | None = None) -> float:
        """L = sum dH * H in fp64."""
        B, K, C, _ = _dims(inp)
        if fwd is None:
            fwd = self.forward(inp)
        return self.lib.cfc_oracle_loss(B, K, C, _p(_f64(fwd["H"])), _p(_f64(inp["dH"])))

    def backward(self, inp: dict, fwd: dict | None = None) -> dict:
        """d_pre [K,B,4,C], dW [4,C,n_in], db [4,C], du [K,B,n_x], dh0 [B,C], all fp64."""
        B, K, C, n_x = _dims(inp)
        if fwd is None:
            fwd = self.forward(inp)
        u, h0, W, ts, dH = (_f64(inp[k]) for k in ("u", "h0", "W", "ts", "dH"))
        H, ff1, ff2, gate = (_f64(fwd[k]) for k in ("H", "ff1", "ff2", "gate"))
        d_pre = np.empty((K, B, 4, C))
        dW = np.empty((4, C, n_x + C))
        db = np.empty((4, C))
        du = np.empty((K, B, n_x))
        dh0 = np.empty((B, C))
        rc = self.lib.cfc_oracle_backward(B, K, C, n_x, _p(u), _p(h0), _p(W), _p(ts), _p(H),
                                          _p(ff1), _p(ff2), _p(gate), _p(dH), _p(d_pre),
                                          _p(dW), _p(db), _p(du), _p(dh0))
        if rc != 0:
            raise ValueError(f"cfc_oracle_backward failed: {rc}")
        return {"d_pre": d_pre, "dW": dW, "db": db, "du": du, "dh0": dh0}

    def reduce_axis0(self, per_batch) -> np.ndarray:
        """out[n] = sum_r per_batch[r, n] in fp64, rows in index order."""
        a = _f64(per_batch)
        n_batch, n_tail = a.shape
        out = np.empty(n_tail)
        rc = self.lib.cfc_oracle_reduce_axis0(n_batch, n_tail, _p(a), _p(out))
        if rc != 0:
            raise ValueError(f"cfc_oracle_reduce_axis0 failed: {rc}")
        return out

    def step(self, inp: dict) -> dict:
        """Forward then backward: every output of one K-loop training step."""
        fwd = self.forward(inp)
        out = dict(fwd)
        out.update(self.backward(inp, fwd))
        return out


def default() -> OracleLib:
    """The oracle built from ``cfc_oracle.c`` (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(inp: dict):
    K, B, n_x = inp["u"].shape
    C = inp["h0"].shape[1]
    return B, K, C, n_x


def forward(inp: dict) -> dict:
    return default().forward(inp)


def loss(inp: dict, fwd: dict | None = None) -> float:
    return default().loss(inp, fwd)


def backward(inp: dict, fwd: dict | None = None) -> dict:
    return default().backward(inp, fwd)


def reduce_axis0(per_batch) -> np.ndarray:
    return default().reduce_axis0(per_batch)


def step(inp: dict) -> dict:
    return default().step(inp)


FP32_NORMAL_MIN = 2.0 ** -126


def rel_err(x, y, floor: float = FP32_NORMAL_MIN) -> float:
    """max|x - y| / max(max|y|, floor) over a whole tensor (the parity metric).

    The floor is fp32's smallest normal number: a tensor whose exact values all lie below
    fp32's normal range (for instance dh0 after a hundred decaying steps) cannot be carried with
    relative precision by an fp32 computation, so it is compared in absolute terms there.
    """
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if y.size == 0:
        return 0.0
    den = max(float(np.max(np.abs(y))), floor)
    return float(np.max(np.abs(x - y))) / den
