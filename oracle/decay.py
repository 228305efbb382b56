"""fp64 CPU oracle of the pages' leaky (tau-decay) cell: forward, BPTT, every gradient.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this package.

The arithmetic lives in ``decay_oracle.c`` (plain C, fp64, single thread); this module builds
it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import compile_source

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decay_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libdecay_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(inp: dict):
    K, B, n_x = inp["x"].shape
    C = inp["h0"].shape[1]
    return B, K, C, n_x


class DecayOracle:
    """ctypes view of one build of the tau-decay oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.cfc_decay_oracle_forward.argtypes = [i] * 4 + [dp] * 8
        lib.cfc_decay_oracle_forward.restype = i
        lib.cfc_decay_oracle_backward.argtypes = [i] * 4 + [dp] * 14
        lib.cfc_decay_oracle_backward.restype = i
        lib.cfc_decay_oracle_loss.argtypes = [i, i, i, dp, dp]
        lib.cfc_decay_oracle_loss.restype = ctypes.c_double
        self.lib = lib

    def forward(self, inp: dict) -> dict:
        """H [K,B,C] and E = tanh(a) [K,B,C], fp64."""
        B, K, C, n_x = _dims(inp)
        x, h0, W, b, tau, ts = (_f64(inp[k]) for k in ("x", "h0", "W", "b", "tau", "ts"))
        H = np.empty((K, B, C))
        E = np.empty((K, B, C))
        rc = self.lib.cfc_decay_oracle_forward(B, K, C, n_x, _p(x), _p(h0), _p(W), _p(b),
                                               _p(tau), _p(ts), _p(H), _p(E))
        if rc != 0:
            raise ValueError(f"cfc_decay_oracle_forward failed: {rc}")
        return {"H": H, "E": E}

    def loss(self, inp: dict, fwd: dict | None = None) -> float:
        B, K, C, _ = _dims(inp)
        if fwd is None:
            fwd = self.forward(inp)
        return self.lib.cfc_decay_oracle_loss(B, K, C, _p(_f64(fwd["H"])), _p(_f64(inp["dH"])))

    def backward(self, inp: dict, fwd: dict | None = None) -> dict:
        """da [K,B,C], dW [C,n_in], db [C], dtau [C], dx [K,B,n_x], dh0 [B,C], fp64."""
        B, K, C, n_x = _dims(inp)
        if fwd is None:
            fwd = self.forward(inp)
        x, h0, W, tau, ts, dH = (_f64(inp[k]) for k in ("x", "h0", "W", "tau", "ts", "dH"))
        H, E = _f64(fwd["H"]), _f64(fwd["E"])
        out = {"da": np.empty((K, B, C)), "dW": np.empty((C, n_x + C)), "db": np.empty(C),
               "dtau": np.empty(C), "dx": np.empty((K, B, n_x)), "dh0": np.empty((B, C))}
        rc = self.lib.cfc_decay_oracle_backward(
            B, K, C, n_x, _p(x), _p(h0), _p(W), _p(tau), _p(ts), _p(H), _p(E), _p(dH),
            _p(out["da"]), _p(out["dW"]), _p(out["db"]), _p(out["dtau"]), _p(out["dx"]),
            _p(out["dh0"]))
        if rc != 0:
            raise ValueError(f"cfc_decay_oracle_backward failed: {rc}")
        return out

    def step(self, inp: dict) -> dict:
        fwd = self.forward(inp)
        out = dict(fwd)
        out.update(self.backward(inp, fwd))
        return out


def default() -> DecayOracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = DecayOracle(build())
    return _lib


def step(inp: dict) -> dict:
    return default().step(inp)
