"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.OracleLib`` (the real build, or a test's mutated
copy) and returns ``(ok, detail)``.  ``test_oracle_pins`` requires every pin to hold on the real
oracle; ``test_oracle_mutants`` requires every planted mistake to break at least one pin.

What each pin leans on:
  * finite differences  -- the backward pass is the gradient of the forward's loss L = sum dH*H;
  * torch.nn.RNN        -- with the time gates fixed at sigmoid(-50) ~ 0 (or +50 ~ 1) the cell
                           is h = tanh(W1 z + b1) (or W2, b2): a textbook Elman RNN whose forward
                           and autograd backward come from the library;
  * torch autograd      -- library derivatives (fp64) of the cell's forward written with
                           torch ops, against the oracle's hand-derived backward;
  * invariants          -- batch rows are independent (batch gradient = sum of per-row
                           gradients, a permutation of the rows permutes the outputs);
  * special cases       -- ts = 0 removes the time-a gradient exactly; a K=1 scalar case.
"""
from __future__ import annotations

import math

import numpy as np

from recurrent_cfc_cell_gb300 import inputs

GRAD_KEYS = ("dW", "db", "du", "dh0")


def _rel(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    den = float(np.max(np.abs(y)))
    num = float(np.max(np.abs(x - y)))
    return num if den == 0.0 else num / den


def _as64(inp: dict) -> dict:
    return {k: np.array(v, dtype=np.float64) for k, v in inp.items()}


def fd_case() -> dict:
    """B=2, K=3, n_x=2, C=3 with nonzero biases and h0 and ts ~ U(0.5, 2)."""
    return _as64(inputs.make_inputs(inputs.custom(B=2, K=3, n_x=2, C=3, seed=11,
                                                  bias_std=0.3, h0_std=0.5)))


def finite_difference_grads(lib, inp: dict, h: float = 1e-5) -> dict:
    """Central differences of L w.r.t. every entry of W, b, u and h0 (fp64)."""
    out = {}
    for key, name in (("W", "dW"), ("b", "db"), ("u", "du"), ("h0", "dh0")):
        arr = inp[key]
        g = np.empty_like(arr)
        flat = arr.reshape(-1)
        gflat = g.reshape(-1)
        for e in range(flat.size):
            keep = flat[e]
            flat[e] = keep + h
            lp = lib.loss(inp)
            flat[e] = keep - h
            lm = lib.loss(inp)
            flat[e] = keep
            gflat[e] = (lp - lm) / (2.0 * h)
        out[name] = g
    return out


def pin_finite_difference(lib, inp: dict | None = None, tol: float = 1e-6):
    inp = fd_case() if inp is None else inp
    an = lib.backward(inp)
    fd = finite_difference_grads(lib, inp)
    errs = {k: _rel(an[k], fd[k]) for k in GRAD_KEYS}
    return all(e <= tol for e in errs.values()), errs


def _rnn_limit_case(active: int, seed: int = 5) -> dict:
    """Only gate ``active`` (0: ff1, 1: ff2) matters: Wa = Wb = 0, ba = 0, bb = -/+50."""
    inp = _as64(inputs.make_inputs(inputs.custom(B=3, K=5, n_x=4, C=6, seed=seed,
                                                 bias_std=0.2, h0_std=0.3)))
    inp["W"][2:] = 0.0
    inp["b"][2] = 0.0
    inp["b"][3] = -50.0 if active == 0 else 50.0
    return inp


def pin_rnn_limit(lib, active: int, tol: float = 1e-12):
    """Gate pinned shut (active=0) or open (active=1): compare with torch.nn.RNN (tanh)."""
    import torch

    inp = _rnn_limit_case(active)
    K, B, n_x = inp["u"].shape
    C = inp["h0"].shape[1]
    Wg = torch.tensor(inp["W"][active])
    bg = torch.tensor(inp["b"][active])
    rnn = torch.nn.RNN(n_x, C, nonlinearity="tanh", bias=True).double()
    with torch.no_grad():
        rnn.weight_ih_l0.copy_(Wg[:, :n_x])
        rnn.weight_hh_l0.copy_(Wg[:, n_x:])
        rnn.bias_ih_l0.copy_(bg)
        rnn.bias_hh_l0.zero_()
    x = torch.tensor(inp["u"], requires_grad=True)
    h0 = torch.tensor(inp["h0"][None], requires_grad=True)
    Ht, _ = rnn(x, h0)
    (Ht * torch.tensor(inp["dH"])).sum().backward()

    o = lib.step(inp)
    errs = {
        "H": _rel(o["H"], Ht.detach().numpy()),
        "dW_in": _rel(o["dW"][active][:, :n_x], rnn.weight_ih_l0.grad.numpy()),
        "dW_rec": _rel(o["dW"][active][:, n_x:], rnn.weight_hh_l0.grad.numpy()),
        "db": _rel(o["db"][active], rnn.bias_ih_l0.grad.numpy()),
        "du": _rel(o["du"], x.grad.numpy()),
        "dh0": _rel(o["dh0"], h0.grad.numpy()[0]),
    }
    ok = all(e <= tol for e in errs.values())
    # The other branch and both time gates carry no gradient in this limit.
    idle = [g for g in range(4) if g != active]
    scale = max(float(np.max(np.abs(o["dW"][active]))), 1e-300)
    errs["idle_dW"] = max(float(np.max(np.abs(o["dW"][g]))) for g in idle) / scale
    errs["idle_db"] = max(float(np.max(np.abs(o["db"][g]))) for g in idle) / scale
    ok = ok and errs["idle_dW"] <= 1e-15 and errs["idle_db"] <= 1e-15
    return ok, errs


def pin_autograd(lib, tol: float = 1e-12):
    """Gradients from torch autograd (fp64) of L for the cell written with torch ops."""
    import torch

    inp = _as64(inputs.make_inputs(inputs.custom(B=2, K=5, n_x=3, C=4, seed=23,
                                                 bias_std=0.3, h0_std=0.5)))
    K, B, n_x = inp["u"].shape
    t = {k: torch.tensor(v, requires_grad=k in ("u", "h0", "W", "b")) for k, v in inp.items()}
    h = t["h0"]
    L = torch.zeros((), dtype=torch.float64)
    for s in range(K):
        z = torch.cat([t["u"][s], h], dim=1)                      # [B, n_in]
        P = torch.einsum("gik,bk->gbi", t["W"], z) + t["b"][:, None, :]
        gate = torch.sigmoid(P[2] * t["ts"][s][:, None] + P[3])
        h = torch.tanh(P[0]) * (1 - gate) + gate * torch.tanh(P[1])
        L = L + (t["dH"][s] * h).sum()
    L.backward()
    ref = {"dW": t["W"].grad.numpy(), "db": t["b"].grad.numpy(), "du": t["u"].grad.numpy(),
           "dh0": t["h0"].grad.numpy()}
    o = lib.backward(inp)
    errs = {k: _rel(o[k], ref[k]) for k in GRAD_KEYS}
    return all(e <= tol for e in errs.values()), errs


def pin_batch_sum(lib, tol: float = 1e-12):
    """Rows are independent: batch gradient = sum of B=1 gradients; per-row outputs match."""
    inp = _as64(inputs.make_inputs(inputs.custom(B=3, K=4, n_x=3, C=5, seed=31)))
    full = lib.step(inp)
    B = inp["h0"].shape[0]
    acc_dW = np.zeros_like(full["dW"])
    acc_db = np.zeros_like(full["db"])
    errs = {"H": 0.0, "du": 0.0, "dh0": 0.0}
    for b in range(B):
        one = {"u": inp["u"][:, b:b + 1], "h0": inp["h0"][b:b + 1], "W": inp["W"],
               "b": inp["b"], "ts": inp["ts"][:, b:b + 1], "dH": inp["dH"][:, b:b + 1]}
        o = lib.step(one)
        acc_dW += o["dW"]
        acc_db += o["db"]
        errs["H"] = max(errs["H"], _rel(full["H"][:, b], o["H"][:, 0]))
        errs["du"] = max(errs["du"], _rel(full["du"][:, b], o["du"][:, 0]))
        errs["dh0"] = max(errs["dh0"], _rel(full["dh0"][b], o["dh0"][0]))
    errs["dW"] = _rel(full["dW"], acc_dW)
    errs["db"] = _rel(full["db"], acc_db)
    return all(e <= tol for e in errs.values()), errs


def pin_permutation(lib, tol: float = 1e-12):
    """Permuting batch rows permutes H, du, dh0 and leaves dW, db unchanged."""
    inp = _as64(inputs.make_inputs(inputs.custom(B=4, K=3, n_x=3, C=4, seed=41)))
    perm = np.array([2, 0, 3, 1])
    pin = {"u": inp["u"][:, perm], "h0": inp["h0"][perm], "W": inp["W"], "b": inp["b"],
           "ts": inp["ts"][:, perm], "dH": inp["dH"][:, perm]}
    a = lib.step(inp)
    p = lib.step(pin)
    errs = {
        "H": _rel(p["H"], a["H"][:, perm]),
        "du": _rel(p["du"], a["du"][:, perm]),
        "dh0": _rel(p["dh0"], a["dh0"][perm]),
        "dW": _rel(p["dW"], a["dW"]),
        "db": _rel(p["db"], a["db"]),
    }
    return all(e <= tol for e in errs.values()), errs


def pin_ts_zero(lib):
    """ts = 0 removes the time-a pre-activation from the gate: its gradients are exactly 0."""
    inp = _as64(inputs.make_inputs(inputs.custom(B=2, K=4, n_x=3, C=4, seed=51)))
    inp["ts"][:] = 0.0
    o = lib.backward(inp)
    ok = (np.all(o["dW"][2] == 0.0) and np.all(o["db"][2] == 0.0)
          and float(np.max(np.abs(o["dW"][3]))) > 1e-6)
    return bool(ok), {"max|dWa|": float(np.max(np.abs(o["dW"][2]))),
                      "max|dWb|": float(np.max(np.abs(o["dW"][3])))}


def pin_scalar_step(lib, tol: float = 1e-14):
    """K=1, B=1, n_x=1, C=1 forward by hand with math.tanh / math.exp."""
    u, h0, ts = 0.7, -0.3, 1.7
    W = np.array([[[0.5, -0.2]], [[-0.4, 0.9]], [[0.3, 0.6]], [[-0.8, 0.1]]])
    b = np.array([[0.05], [-0.1], [0.2], [-0.3]])
    P = [W[g, 0, 0] * u + W[g, 0, 1] * h0 + b[g, 0] for g in range(4)]
    f1, f2 = math.tanh(P[0]), math.tanh(P[1])
    gt = 1.0 / (1.0 + math.exp(-(P[2] * ts + P[3])))
    h = f1 * (1.0 - gt) + gt * f2
    inp = {"u": np.array([[[u]]]), "h0": np.array([[h0]]), "W": W, "b": b,
           "ts": np.array([[ts]]), "dH": np.array([[[1.0]]])}
    o = lib.forward(inp)
    errs = {"H": abs(o["H"][0, 0, 0] - h), "ff1": abs(o["ff1"][0, 0, 0] - f1),
            "ff2": abs(o["ff2"][0, 0, 0] - f2), "gate": abs(o["gate"][0, 0, 0] - gt)}
    return all(e <= tol for e in errs.values()), errs


def pin_reduce_axis0(lib, tol: float = 1e-13):
    """Axis-0 sum against math.fsum (correctly rounded) and an exactly representable case."""
    rng = np.random.default_rng(61)
    a = rng.normal(0, 1, size=(37, 11))
    out = lib.reduce_axis0(a)
    ref = np.array([math.fsum(a[:, n]) for n in range(a.shape[1])])
    ints = rng.integers(-1000, 1000, size=(50, 7)).astype(np.float64)
    exact = bool(np.all(lib.reduce_axis0(ints) == ints.sum(axis=0)))
    err = _rel(out, ref)
    return err <= tol and exact, {"fsum": err, "exact_ints": exact}


ALL_PINS = {
    "finite_difference": pin_finite_difference,
    "rnn_limit_gate_shut": lambda lib: pin_rnn_limit(lib, 0),
    "rnn_limit_gate_open": lambda lib: pin_rnn_limit(lib, 1),
    "autograd": pin_autograd,
    "batch_sum": pin_batch_sum,
    "permutation": pin_permutation,
    "ts_zero": pin_ts_zero,
    "scalar_step": pin_scalar_step,
    "reduce_axis0": pin_reduce_axis0,
}
