"""One CfC K-loop training step (forward + BPTT + gradients) on the current CUDA device.

``KLoopStep`` owns the outputs and the workspace (allocated once through PyTorch), runs
cfc_forward_backward (cfc_forward then cfc_backward) on one stream, and can capture it into a
CUDA graph so a step
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
        # The forward's own workspace (its exchange buffer at large B), apart from ws so that a
        # forward never overwrites the d_pre a backward left at the head of ws.
        nf = _lib.forward_workspace_bytes(B, K, C, n_x)
        self.fws = torch.empty(nf, dtype=torch.uint8, device=dev) if nf else None
        self.inputs = None
        self.graph = None

    @property
    def d_pre_is_fp32(self) -> bool:
        return self.dw_mode in (_lib.CFC_DW_TF32, _lib.CFC_DW_SIMT_FP32)

    @property
    def d_pre(self) -> torch.Tensor:
        """The head of the workspace, where the backward pass leaves the pre-activation
        gradients (valid after backward), as include/cfc.h lays it out for the mode: fp32
        [K, B, 4, C] for the TF32 and SIMT modes; otherwise the raw bf16 operand rows as int16
        [K, B, 2, MP] (term, then MP = 4C rounded up to 8 values: hi, lo)."""
        K, B, C = self.K, self.B, self.C
        if self.d_pre_is_fp32:
            return self.ws[: 16 * K * B * C].view(torch.float32).view(K, B, 4, C)
        mp = _lib.dpre_operand_pitch(C, self.dw_mode)
        return self.ws[: 4 * K * B * mp].view(torch.int16).view(K, B, 2, mp)

    @property
    def d_pre_fp32_view(self) -> torch.Tensor:
        """The head of the workspace viewed as fp32 [K, B, 4, C]: where the stage entry points
        (cfc_backward_recurrence_ws, then cfc_weight_grad) may keep an fp32 d_pre in place."""
        n = self.K * self.B * 4 * self.C
        return self.ws[: 4 * n].view(torch.float32).view(self.K, self.B, 4, self.C)

    def bind(self, u, h0, W, b, ts, dH) -> "KLoopStep":
        """Use these device tensors as the step's inputs (kept by reference)."""
        self.inputs = dict(u=u, h0=h0, W=W, b=b, ts=ts, dH=dH)
        return self

    def forward(self, stream=None) -> None:
        i = self.inputs
        _lib.cfc_forward(i["u"], i["h0"], i["W"], i["b"], i["ts"], self.H, self.cache,
                         ws=self.fws, stream=stream)

    def backward(self, stream=None) -> None:
        i = self.inputs
        _lib.cfc_backward(i["dH"], i["u"], i["h0"], i["W"], i["ts"], self.H, self.cache,
                          self.dW, self.db, self.du, self.dh0, self.ws, self.dw_mode,
                          stream=stream)

    def run(self, stream=None) -> None:
        """Forward then backward in one cfc_forward_backward call, enqueued on ``stream``
        (default: current stream)."""
        i = self.inputs
        _lib.cfc_forward_backward(i["u"], i["h0"], i["W"], i["b"], i["ts"], i["dH"], self.H,
                                  self.cache, self.dW, self.db, self.du, self.dh0, self.ws,
                                  self.dw_mode, stream=stream)

    # ---- host staging: one pinned buffer of inputs in, one of gradients out ----------------
    @staticmethod
    def _pack(shapes: dict, device, pinned: bool):
        """One flat fp32 buffer holding every shape at a 256-byte-aligned offset, and its views."""
        off, offs = 0, {}
        for k, shp in shapes.items():
            offs[k] = off
            n = 1
            for d in shp:
                n *= d
            off += (n + 63) // 64 * 64
        buf = torch.empty(off, dtype=torch.float32, device=device)
        if pinned:
            buf = buf.pin_memory()
        views = {}
        for k, shp in shapes.items():
            n = 1
            for d in shp:
                n *= d
            views[k] = buf[offs[k]: offs[k] + n].view(*shp)
        return buf, views

    def stage_host(self) -> "KLoopStep":
        """Give the step packed input and gradient buffers on the device, each with a pinned
        host twin, so one copy brings a step's inputs in and one copy takes its gradients out
        (capture(with_host_io=True) puts both copies in the step's graph).  Fill
        ``host_in[name]``; read ``host_out[name]`` after the step."""
        B, K, C, n_x, n_in = self.B, self.K, self.C, self.n_x, self.n_in
        shapes_in = {"u": (K, B, n_x), "h0": (B, C), "W": (4, C, n_in), "b": (4, C),
                     "ts": (K, B), "dH": (K, B, C)}
        shapes_out = {"dW": (4, C, n_in), "db": (4, C), "dh0": (B, C)}
        if self.du is not None:
            shapes_out["du"] = (K, B, n_x)
        self._dev_in, self.inputs = self._pack(shapes_in, self.device, False)
        self._host_in_buf, self.host_in = self._pack(shapes_in, "cpu", True)
        self._dev_out, outs = self._pack(shapes_out, self.device, False)
        self._host_out_buf, self.host_out = self._pack(shapes_out, "cpu", True)
        self.dW, self.db, self.dh0 = outs["dW"], outs["db"], outs["dh0"]
        if self.du is not None:
            self.du = outs["du"]
        self.graph = None
        return self

    def io_bytes(self) -> tuple[int, int]:
        """Bytes of real tensor data one staged step copies in and out."""
        n_in = sum(v.numel() for v in self.host_in.values()) * 4
        n_out = sum(v.numel() for v in self.host_out.values()) * 4
        return n_in, n_out

    def run_with_host_io(self, stream=None) -> None:
        """Inputs in from the pinned host buffer, the step, gradients out to it.  Both copies
        are the library's copy kernel (cfc_copy), which reads and writes the pinned host memory
        directly: on GB300 a graph step with it took 122 us at B=32, K=64, C=128 against 132 us
        with copy-engine transfers of the same 1.8 MB in and 0.8 MB out."""
        _lib.copy(self._host_in_buf, self._dev_in, stream)
        self.run(stream)
        _lib.copy(self._dev_out, self._host_out_buf, stream)

    def capture(self, with_host_io: bool = False) -> torch.cuda.CUDAGraph:
        """Capture run() (or run_with_host_io()) into a CUDA graph (one eager run first sets
        kernel attributes)."""
        fn = self.run_with_host_io if with_host_io else self.run
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
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
