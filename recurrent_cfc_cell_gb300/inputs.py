"""Seeded synthetic inputs for the CfC K-loop (forward + BPTT + weight gradient).

This module only draws random numbers; it holds none of the cell's arithmetic. Both the
fp64 oracle (test infrastructure) and the CUDA path consume the fp32 arrays it returns.

Workloads. The K-loop parallelization spec (page "K-loop Parallelization -- Block-per-Batch
Kernel Refactor", section "Problem") runs the cell at batch B=32 over a 64-step K-loop with
hidden width 128 on an L40S; its data set is private, so every input here is synthetic with
the shapes and value distributions listed in ``CONFIGS``.

Readings of the workload text (each is a plain reading where the text is open):
  * "N(0, s)" is a normal with standard deviation s.
  * weights are U(-1/sqrt(n_in), 1/sqrt(n_in)), one [C, n_in] matrix per gate.
  * "10% of u entries exactly 0" zeroes exactly floor(0.1 * K*B*n_x) entries, chosen by a
    seeded permutation.  Only the wide-state workload states it, so only it has zeros.
  * "dL/dh_t nonzero only at the last 8 steps" means t in [K-8, K).
  * the draw order is fixed: W1, W2, Wa, Wb, b1, b2, ba, bb, h0, u, zero mask, ts, dH; each
    value is drawn in fp64 by numpy's PCG64 and rounded to fp32.

Layouts (row-major, last index fastest):
  u [K, B, n_x], h0 [B, C], W [4, C, n_x + C] (gate order ff1, ff2, time-a, time-b; the
  columns follow z = [u_t ; h_{t-1}]), b [4, C], ts [K, B], dH [K, B, C].
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value distributions of one synthetic K-loop workload."""

    name: str
    B: int
    K: int
    n_x: int
    C: int
    seed: int
    bias_std: float = 0.01
    h0_std: float = 0.1
    ts_range: tuple | None = (0.5, 2.0)  # None: ts = 1.0 everywhere
    u_zero_frac: float = 0.0
    dH_last: int | None = None  # None: upstream gradient at every step

    @property
    def n_in(self) -> int:
        return self.n_x + self.C

    @property
    def units(self) -> int:
        """Sequence-steps processed by one pass (B * K)."""
        return self.B * self.K

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "K": self.K, "n_x": self.n_x, "C": self.C,
                "seed": self.seed}


# The five workloads: tiny, the pages' shape (B=32, K=64, C=128), wider state, larger batch,
# throughput stress.
CONFIGS = [
    Workload("tiny_B4_K8_nx16_C32", B=4, K=8, n_x=16, C=32, seed=0,
             bias_std=0.0, h0_std=0.0, ts_range=None),
    Workload("pages_B32_K64_nx48_C128", B=32, K=64, n_x=48, C=128, seed=1),
    Workload("wide_B32_K64_nx64_C256", B=32, K=64, n_x=64, C=256, seed=2, u_zero_frac=0.1),
    Workload("batch_B256_K64_nx48_C128", B=256, K=64, n_x=48, C=128, seed=3),
    Workload("stress_B2048_K128_nx64_C256", B=2048, K=128, n_x=64, C=256, seed=4,
             ts_range=(0.1, 4.0), dH_last=8),
]


def custom(B: int, K: int, n_x: int, C: int, seed: int = 7, **kw) -> Workload:
    """An ad-hoc workload with the distributions of the pages' shape (for edge cases)."""
    return Workload(f"custom_B{B}_K{K}_nx{n_x}_C{C}", B=B, K=K, n_x=n_x, C=C, seed=seed, **kw)


def make_inputs(w: Workload) -> dict:
    """Draw u, h0, W, b, ts, dH for workload ``w`` (fp32, C-contiguous)."""
    rng = np.random.default_rng(w.seed)
    B, K, n_x, C, n_in = w.B, w.K, w.n_x, w.C, w.n_in
    lim = 1.0 / math.sqrt(n_in)
    W = np.empty((4, C, n_in), dtype=np.float32)
    for g in range(4):
        W[g] = rng.uniform(-lim, lim, size=(C, n_in))
    b = np.zeros((4, C), dtype=np.float32)
    if w.bias_std > 0:
        for g in range(4):
            b[g] = rng.normal(0.0, w.bias_std, size=C)
    if w.h0_std > 0:
        h0 = rng.normal(0.0, w.h0_std, size=(B, C)).astype(np.float32)
    else:
        h0 = np.zeros((B, C), dtype=np.float32)
    u = rng.normal(0.0, 1.0, size=(K, B, n_x)).astype(np.float32)
    if w.u_zero_frac > 0:
        n_zero = int(math.floor(w.u_zero_frac * u.size))
        idx = rng.permutation(u.size)[:n_zero]
        u.reshape(-1)[idx] = 0.0
    if w.ts_range is None:
        ts = np.ones((K, B), dtype=np.float32)
    else:
        ts = rng.uniform(w.ts_range[0], w.ts_range[1], size=(K, B)).astype(np.float32)
    dH = np.zeros((K, B, C), dtype=np.float32)
    if w.dH_last is None:
        dH[:] = rng.normal(0.0, 1.0, size=(K, B, C))
    else:
        last = min(w.dH_last, K)
        dH[K - last:] = rng.normal(0.0, 1.0, size=(last, B, C))
    return {"u": np.ascontiguousarray(u), "h0": np.ascontiguousarray(h0),
            "W": np.ascontiguousarray(W), "b": np.ascontiguousarray(b),
            "ts": np.ascontiguousarray(ts), "dH": np.ascontiguousarray(dH)}


# ---- the pages' own leaky (tau-decay) cell ----
#
# Its backward names grad_w_in [B,128,128], grad_w_rec [B,128,128], grad_b and grad_tau [B,128]
# (page "K-loop Parallelization -- Block-per-Batch Kernel Refactor", section "Per-Kernel
# Breakdown"), so the pages' shape is 128 inputs and 128 hidden units at B = 32 over 64 steps.
# Readings: W = [W_in | W_rec] is one [C, n_x + C] matrix, U(-1/sqrt(n_in), 1/sqrt(n_in)) like
# the four-gate cell's; tau (a time constant per hidden unit, positive) is U(0.5, 4); ts, x, h0,
# b and dH follow the four-gate workloads.  Draw order: W, b, tau, h0, x, ts, dH.
# Layouts: x [K, B, n_x], h0 [B, C], W [C, n_x + C], b [C], tau [C], ts [K, B], dH [K, B, C].

@dataclasses.dataclass(frozen=True)
class DecayWorkload:
    """Shape and value distributions of one synthetic workload of the tau-decay cell."""

    name: str
    B: int
    K: int
    n_x: int
    C: int
    seed: int
    tau_range: tuple = (0.5, 4.0)
    ts_range: tuple = (0.5, 2.0)

    @property
    def n_in(self) -> int:
        return self.n_x + self.C

    @property
    def units(self) -> int:
        return self.B * self.K

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "K": self.K, "n_x": self.n_x, "C": self.C,
                "seed": self.seed, "cell": "tau-decay"}


DECAY_CONFIGS = [
    DecayWorkload("decay_tiny_B4_K8_nx16_C32", B=4, K=8, n_x=16, C=32, seed=10),
    DecayWorkload("decay_pages_B32_K64_nx128_C128", B=32, K=64, n_x=128, C=128, seed=11),
    DecayWorkload("decay_batch_B256_K64_nx128_C128", B=256, K=64, n_x=128, C=128, seed=12),
]


def decay_custom(B: int, K: int, n_x: int, C: int, seed: int = 17, **kw) -> DecayWorkload:
    return DecayWorkload(f"decay_custom_B{B}_K{K}_nx{n_x}_C{C}", B=B, K=K, n_x=n_x, C=C,
                         seed=seed, **kw)


def make_decay_inputs(w: DecayWorkload) -> dict:
    """Draw x, h0, W, b, tau, ts, dH for the tau-decay workload ``w`` (fp32, C-contiguous)."""
    rng = np.random.default_rng(w.seed)
    B, K, n_x, C, n_in = w.B, w.K, w.n_x, w.C, w.n_in
    lim = 1.0 / math.sqrt(n_in)
    W = rng.uniform(-lim, lim, size=(C, n_in)).astype(np.float32)
    b = rng.normal(0.0, 0.01, size=C).astype(np.float32)
    tau = rng.uniform(w.tau_range[0], w.tau_range[1], size=C).astype(np.float32)
    h0 = rng.normal(0.0, 0.1, size=(B, C)).astype(np.float32)
    x = rng.normal(0.0, 1.0, size=(K, B, n_x)).astype(np.float32)
    ts = rng.uniform(w.ts_range[0], w.ts_range[1], size=(K, B)).astype(np.float32)
    dH = rng.normal(0.0, 1.0, size=(K, B, C)).astype(np.float32)
    return {"x": x, "h0": h0, "W": W, "b": b, "tau": tau, "ts": ts, "dH": dH}
