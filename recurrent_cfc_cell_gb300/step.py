"""One CfC K-loop training step (forward + BPTT + gradients) on the current CUDA device.

``KLoopStep`` owns the outputs and the workspace (allocated once through PyTorch), runs
cfc_forward then cfc_backward on one stream, and can capture both into a CUDA graph so a step
is a single graph replay (the spec's "CUDA Graph capture / replay" of the training step,
page "K-loop Parallelization -- Block-per-Batch Kernel Refactor", section "Trainer Wiring").
"""
from __future__ import annotations

import torch

from . import _lib


class KLoopStep:
    """Buffers and launches of one (B, K, C, n_x) K-loop step."""

    def __init__(self, B: int, K: int, C: int, n_x: int, dw_mode: int = _lib.CFC_DW_ACCURATE,
                 device: torch.device | str | None = None, with_du: bool = True):
        self.B, self.K, self.C, self.n_x = B, K, C, n_x
        self.n_in = n_x + C
        self.dw_mode = dw_mode
        dev = torch.device(device) if device is not None else torch.device("cuda",
                                                                            torch.cuda.current_device())
        f32 = dict(dtype=torch.float32, device=dev)
        self.device = dev
        self.H = torch.empty((K, B, C), **f32)
        self.cache = torch.empty((K, B, 3, C), **f32)
        self.dW = torch.empty((4, C, self.n_in), **f32)
        self.db = torch.empty((4, C), **f32)
        self.du = torch.empty((K, B, n_x), **f32) if with_du else None
        self.dh0 = torch.empty((B, C), **f32)
        self.ws = torch.empty(_lib.workspace_bytes(B, K, C, n_x, dw_mode), dtype=torch.uint8,
                              device=dev)
        self.inputs = None
        self.graph = None

    @property
    def d_pre(self) -> torch.Tensor:
        """Pre-activation gradients [K, B, 4, C] (head of the workspace, valid after backward)."""
        n = self.K * self.B * 4 * self.C
        return self.ws[: 4 * n].view(torch.float32).view(self.K, self.B, 4, self.C)

    def bind(self, u, h0, W, b, ts, dH) -> "KLoopStep":
        """Use these device tensors as the step's inputs (kept by reference)."""
        self.inputs = dict(u=u, h0=h0, W=W, b=b, ts=ts, dH=dH)
        return self

    def forward(self, stream=None) -> None:
        i = self.inputs
        _lib.cfc_forward(i["u"], i["h0"], i["W"], i["b"], i["ts"], self.H, self.cache,
                         stream=stream)

    def backward(self, stream=None) -> None:
        i = self.inputs
        _lib.cfc_backward(i["dH"], i["u"], i["h0"], i["W"], i["ts"], self.H, self.cache,
                          self.dW, self.db, self.du, self.dh0, self.ws, self.dw_mode,
                          stream=stream)

    def run(self, stream=None) -> None:
        """Forward then backward, enqueued on ``stream`` (default: current stream)."""
        self.forward(stream)
        self.backward(stream)

    def capture(self) -> torch.cuda.CUDAGraph:
        """Capture run() into a CUDA graph (one eager run first sets kernel attributes)."""
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self) -> None:
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def outputs(self) -> dict:
        out = {"H": self.H, "cache": self.cache, "dW": self.dW, "db": self.db,
               "dh0": self.dh0, "d_pre": self.d_pre}
        if self.du is not None:
            out["du"] = self.du
        return out


def to_device(inp: dict, device=None) -> dict:
    """numpy fp32 inputs -> contiguous CUDA tensors."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return {k: torch.from_numpy(v).to(dev).contiguous() for k, v in inp.items()}
