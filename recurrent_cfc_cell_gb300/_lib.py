"""ctypes binding of libcfc.so (include/cfc.h): argument marshalling only.

Every function takes torch tensors that already live on the current CUDA device, checks
dtype / contiguity / shape on the host, passes raw pointers and the current stream to the C
entry point of the same name and raises ``CfcError`` on a non-zero status.  All computation
happens in the library's CUDA kernels.  If the library has not been built (or fails to load)
importing it raises, so nothing can silently run elsewhere.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libcfc.so")

CFC_OK = 0
CFC_DW_ACCURATE = 0   # tensor cores, two bf16 terms per operand (three products per step)
CFC_DW_BF16 = 1       # tensor cores, one bf16 product per step
CFC_DW_TF32 = 2       # tensor cores, one tf32 product per step
CFC_DW_SIMT_FP32 = 3  # CUDA-core fp32
DW_MODES = (CFC_DW_ACCURATE, CFC_DW_BF16, CFC_DW_TF32, CFC_DW_SIMT_FP32)


def dpre_operand_pitch(C: int, dw_mode: int) -> int:
    """bf16 values per term in a d_pre row of the workspace head (modes ACCURATE and BF16), as
    include/cfc.h documents: 4C rounded up to a multiple of 8."""
    return (4 * C + 7) // 8 * 8

# Public C symbols declared in include/cfc.h (checked by the test suite).
EXPORTED = ("cfc_workspace_bytes", "cfc_forward", "cfc_backward", "cfc_backward_recurrence",
            "cfc_weight_grad", "reduce_axis0", "cfc_error_string", "cfc_device_status",
            "cfc_backward_noalloc", "cfc_input_projection", "cfc_forward_recurrence",
            "cfc_step_launches", "cfc_forward_backward", "cfc_bptt_workspace_bytes",
            "cfc_backward_recurrence_ws", "cfc_wait_self_test", "cfc_probe_fma",
            "cfc_probe_l2_read", "cfc_forward_bf16_workspace_bytes", "cfc_forward_bf16",
            "cfc_backward_bf16", "cfc_decay_forward", "cfc_decay_workspace_bytes",
            "cfc_decay_backward", "cfc_forward_workspace_bytes", "cfc_copy")
CFC_ERR_SCRATCH_LIMIT = -10
NOALLOC_SCRATCH_BYTES = 32 << 20  # size of cfc_backward_noalloc's built-in device scratch


class CfcError(RuntimeError):
    def __init__(self, func: str, code: int, text: str):
        super().__init__(f"{func} failed: {code} ({text})")
        self.code = code


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libcfc.so (raises if it is missing: build it with recurrent_cfc_cell_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libcfc.so not built ({p}); run python -m recurrent_cfc_cell_gb300.build")
    lib = ctypes.CDLL(p)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.cfc_workspace_bytes.argtypes = [i, i, i, i, i, ctypes.POINTER(sz)]
    lib.cfc_workspace_bytes.restype = i
    lib.cfc_forward.argtypes = [vp] * 5 + [i] * 4 + [vp, vp, vp, sz, vp]
    lib.cfc_forward.restype = i
    lib.cfc_backward.argtypes = [vp] * 7 + [i] * 4 + [vp] * 5 + [sz, i, vp]
    lib.cfc_backward.restype = i
    lib.cfc_forward_backward.argtypes = [vp] * 6 + [i] * 4 + [vp] * 7 + [sz, i, vp]
    lib.cfc_forward_backward.restype = i
    lib.cfc_backward_recurrence.argtypes = [vp] * 4 + [i] * 4 + [vp, vp, vp]
    lib.cfc_backward_recurrence.restype = i
    lib.cfc_bptt_workspace_bytes.argtypes = [i] * 4 + [vp]
    lib.cfc_bptt_workspace_bytes.restype = i
    lib.cfc_backward_recurrence_ws.argtypes = [vp] * 4 + [i] * 4 + [vp, vp, vp, sz, vp]
    lib.cfc_backward_recurrence_ws.restype = i
    lib.cfc_weight_grad.argtypes = [vp] * 5 + [i] * 4 + [vp] * 4 + [sz, i, vp]
    lib.cfc_weight_grad.restype = i
    lib.reduce_axis0.argtypes = [vp, i, i, vp, vp]
    lib.reduce_axis0.restype = i
    lib.cfc_input_projection.argtypes = [vp] * 3 + [i] * 4 + [vp, vp, vp]
    lib.cfc_input_projection.restype = i
    lib.cfc_forward_recurrence.argtypes = [vp] * 3 + [i] * 4 + [vp, vp, vp, sz, vp]
    lib.cfc_forward_recurrence.restype = i
    lib.cfc_step_launches.argtypes = [i] * 6 + [ctypes.POINTER(i)]
    lib.cfc_step_launches.restype = i
    lib.cfc_backward_noalloc.argtypes = [vp] * 7 + [i] * 4 + [vp] * 4 + [i, vp]
    lib.cfc_backward_noalloc.restype = i
    lib.cfc_error_string.argtypes = [i]
    lib.cfc_error_string.restype = ctypes.c_char_p
    lib.cfc_device_status.argtypes = [ctypes.POINTER(i)]
    lib.cfc_device_status.restype = i
    lib.cfc_wait_self_test.argtypes = [vp]
    lib.cfc_wait_self_test.restype = i
    dptr = ctypes.POINTER(ctypes.c_double)
    lib.cfc_probe_fma.argtypes = [vp, i, i, dptr, vp]
    lib.cfc_probe_fma.restype = i
    lib.cfc_probe_l2_read.argtypes = [vp, sz, i, vp, i, dptr, vp]
    lib.cfc_probe_l2_read.restype = i
    lib.cfc_forward_bf16_workspace_bytes.argtypes = [i] * 4 + [ctypes.POINTER(sz)]
    lib.cfc_forward_workspace_bytes.argtypes = [i] * 4 + [ctypes.POINTER(sz)]
    lib.cfc_forward_workspace_bytes.restype = i
    lib.cfc_forward_bf16_workspace_bytes.restype = i
    lib.cfc_forward_bf16.argtypes = [vp] * 5 + [i] * 4 + [vp, vp, vp, sz, vp]
    lib.cfc_forward_bf16.restype = i
    lib.cfc_backward_bf16.argtypes = [vp] * 7 + [i] * 4 + [vp] * 5 + [sz, vp]
    lib.cfc_backward_bf16.restype = i
    lib.cfc_decay_forward.argtypes = [vp] * 6 + [i] * 4 + [vp, vp, vp]
    lib.cfc_decay_forward.restype = i
    lib.cfc_decay_workspace_bytes.argtypes = [i] * 4 + [ctypes.POINTER(sz)]
    lib.cfc_decay_workspace_bytes.restype = i
    lib.cfc_decay_backward.argtypes = [vp] * 8 + [i] * 4 + [vp] * 6 + [sz, vp]
    lib.cfc_decay_backward.restype = i
    lib.cfc_copy.argtypes = [vp, vp, sz, vp]
    lib.cfc_copy.restype = i
    if path is None:
        _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().cfc_error_string(int(code)).decode()


def _check(func: str, rc: int) -> None:
    if rc != CFC_OK:
        raise CfcError(func, rc, error_string(rc))


def _ptr(t, name: str, shape=None):
    import torch

    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _ptr16(t, name: str, shape):
    """A contiguous bfloat16 CUDA tensor of the given shape (bf16 H / cache)."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


def _ws(ws):
    import torch

    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("ws must be a contiguous uint8 CUDA tensor")
    return ctypes.c_void_p(ws.data_ptr()), ws.numel()


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(B: int, K: int, C: int, n_x: int, dw_mode: int = CFC_DW_ACCURATE) -> int:
    out = ctypes.c_size_t(0)
    _check("cfc_workspace_bytes",
           load().cfc_workspace_bytes(B, K, C, n_x, dw_mode, ctypes.byref(out)))
    return out.value


def forward_workspace_bytes(B: int, K: int, C: int, n_x: int) -> int:
    out = ctypes.c_size_t(0)
    _check("cfc_forward_workspace_bytes",
           load().cfc_forward_workspace_bytes(B, K, C, n_x, ctypes.byref(out)))
    return out.value


def _fwd_ws(ws, B, K, C, n_x, like):
    """(pointer, bytes) of the forward's workspace: `ws`, or a fresh device buffer when the
    caller gave none and the sizes need one."""
    if ws is None:
        need = forward_workspace_bytes(B, K, C, n_x)
        if need == 0:
            return None, 0, None
        import torch

        ws = torch.empty(need, dtype=torch.uint8, device=like.device)
    p, n = _ws(ws)
    return p, n, ws


def cfc_forward(u, h0, W, b, ts, H, cache, ws=None, stream=None) -> None:
    """H [K,B,C] and cache [K,B,3,C] <- forward recurrence over K steps.  `ws`: a uint8
    device buffer of forward_workspace_bytes() bytes (allocated here when None and needed)."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    wp, wn, _keep = _fwd_ws(ws, B, K, C, n_x, H)
    rc = load().cfc_forward(
        _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)), _ptr(W, "W", (4, C, n_in)),
        _ptr(b, "b", (4, C)), _ptr(ts, "ts", (K, B)), B, K, C, n_x,
        _ptr(H, "H", (K, B, C)), _ptr(cache, "cache", (K, B, 3, C)), wp, wn, _stream(stream))
    _check("cfc_forward", rc)


def cfc_input_projection(u, W, b, H, cache, stream=None) -> None:
    """X = W_u u + b for all steps, written in place into H (ff1) and cache (ff2, ta, tb)."""
    K, B, n_x = u.shape
    C = H.shape[2]
    rc = load().cfc_input_projection(
        _ptr(u, "u", (K, B, n_x)), _ptr(W, "W", (4, C, n_x + C)), _ptr(b, "b", (4, C)),
        B, K, C, n_x, _ptr(H, "H", (K, B, C)), _ptr(cache, "cache", (K, B, 3, C)),
        _stream(stream))
    _check("cfc_input_projection", rc)


def cfc_forward_recurrence(h0, W, ts, H, cache, ws=None, stream=None) -> None:
    """The K-step recurrence on top of the projection left in H / cache (`ws` as for
    cfc_forward)."""
    K, B, C = H.shape
    n_x = W.shape[2] - C
    wp, wn, _keep = _fwd_ws(ws, B, K, C, n_x, H)
    rc = load().cfc_forward_recurrence(
        _ptr(h0, "h0", (B, C)), _ptr(W, "W", (4, C, n_x + C)), _ptr(ts, "ts", (K, B)),
        B, K, C, n_x, _ptr(H, "H", (K, B, C)), _ptr(cache, "cache", (K, B, 3, C)), wp, wn,
        _stream(stream))
    _check("cfc_forward_recurrence", rc)


def step_launches(B: int, K: int, C: int, n_x: int, dw_mode: int = CFC_DW_ACCURATE,
                  with_du: bool = True) -> int:
    """Kernel launches of one cfc_forward + cfc_backward for these sizes."""
    out = ctypes.c_int(0)
    _check("cfc_step_launches",
           load().cfc_step_launches(B, K, C, n_x, dw_mode, int(with_du), ctypes.byref(out)))
    return out.value


def cfc_backward(dH, u, h0, W, ts, H, cache, dW, db, du, dh0, ws,
                 dw_mode: int = CFC_DW_ACCURATE, stream=None) -> None:
    """dW, db, du (optional), dh0 and d_pre (at the head of ws) <- BPTT + contractions."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    import torch

    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("ws must be a contiguous uint8 CUDA tensor")
    rc = load().cfc_backward(
        _ptr(dH, "dH", (K, B, C)), _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)),
        _ptr(W, "W", (4, C, n_in)), _ptr(ts, "ts", (K, B)), _ptr(H, "H", (K, B, C)),
        _ptr(cache, "cache", (K, B, 3, C)), B, K, C, n_x, _ptr(dW, "dW", (4, C, n_in)),
        _ptr(db, "db", (4, C)), _ptr(du, "du", (K, B, n_x)), _ptr(dh0, "dh0", (B, C)),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), dw_mode, _stream(stream))
    _check("cfc_backward", rc)


def cfc_forward_backward(u, h0, W, b, ts, dH, H, cache, dW, db, du, dh0, ws,
                         dw_mode: int = CFC_DW_ACCURATE, stream=None) -> None:
    """One training step: cfc_forward then cfc_backward in one call (the backward recurrence
    launched as a dependent of the forward)."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    import torch

    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("ws must be a contiguous uint8 CUDA tensor")
    rc = load().cfc_forward_backward(
        _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)), _ptr(W, "W", (4, C, n_in)),
        _ptr(b, "b", (4, C)), _ptr(ts, "ts", (K, B)), _ptr(dH, "dH", (K, B, C)), B, K, C, n_x,
        _ptr(H, "H", (K, B, C)), _ptr(cache, "cache", (K, B, 3, C)),
        _ptr(dW, "dW", (4, C, n_in)), _ptr(db, "db", (4, C)), _ptr(du, "du", (K, B, n_x)),
        _ptr(dh0, "dh0", (B, C)), ctypes.c_void_p(ws.data_ptr()), ws.numel(), dw_mode,
        _stream(stream))
    _check("cfc_forward_backward", rc)


def cfc_backward_recurrence(dH, W, ts, cache, d_pre, dh0, stream=None) -> None:
    """d_pre [K,B,4,C] and dh0 [B,C] <- reverse-time recurrence only."""
    K, B, C = dH.shape
    n_x = W.shape[2] - C
    rc = load().cfc_backward_recurrence(
        _ptr(dH, "dH", (K, B, C)), _ptr(W, "W", (4, C, n_x + C)), _ptr(ts, "ts", (K, B)),
        _ptr(cache, "cache", (K, B, 3, C)), B, K, C, n_x, _ptr(d_pre, "d_pre", (K, B, 4, C)),
        _ptr(dh0, "dh0", (B, C)), _stream(stream))
    _check("cfc_backward_recurrence", rc)


def bptt_workspace_bytes(B: int, K: int, C: int, n_x: int) -> int:
    """Workspace bytes cfc_backward_recurrence_ws takes (0: the CUDA-core recurrence runs)."""
    out = ctypes.c_size_t(0)
    _check("cfc_bptt_workspace_bytes",
           load().cfc_bptt_workspace_bytes(B, K, C, n_x, ctypes.byref(out)))
    return int(out.value)


def cfc_backward_recurrence_ws(dH, W, ts, cache, d_pre, dh0, ws=None, stream=None) -> None:
    """As cfc_backward_recurrence, with a workspace (a uint8 CUDA tensor of at least
    bptt_workspace_bytes(B, K, C, n_x) bytes, or None when that is 0) so that large batches
    take the tensor-core recurrence."""
    import torch

    K, B, C = dH.shape
    n_x = W.shape[2] - C
    if ws is None:
        wp, wn = None, 0
    else:
        if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
            raise ValueError("ws must be a contiguous uint8 CUDA tensor")
        wp, wn = ctypes.c_void_p(ws.data_ptr()), ws.numel()
    rc = load().cfc_backward_recurrence_ws(
        _ptr(dH, "dH", (K, B, C)), _ptr(W, "W", (4, C, n_x + C)), _ptr(ts, "ts", (K, B)),
        _ptr(cache, "cache", (K, B, 3, C)), B, K, C, n_x, _ptr(d_pre, "d_pre", (K, B, 4, C)),
        _ptr(dh0, "dh0", (B, C)), wp, wn, _stream(stream))
    _check("cfc_backward_recurrence_ws", rc)


def cfc_weight_grad(d_pre, u, h0, W, H, dW, db, du, ws, dw_mode: int = CFC_DW_ACCURATE,
                    stream=None) -> None:
    """dW, db, du (optional) <- contractions of d_pre (second stage of cfc_backward)."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    rc = load().cfc_weight_grad(
        _ptr(d_pre, "d_pre", (K, B, 4, C)), _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)),
        _ptr(W, "W", (4, C, n_in)), _ptr(H, "H", (K, B, C)), B, K, C, n_x,
        _ptr(dW, "dW", (4, C, n_in)), _ptr(db, "db", (4, C)), _ptr(du, "du", (K, B, n_x)),
        ctypes.c_void_p(ws.data_ptr()), ws.numel(), dw_mode, _stream(stream))
    _check("cfc_weight_grad", rc)


def reduce_axis0(per_batch, out, stream=None) -> None:
    """out[n] <- sum_r per_batch[r, n] (overwrite, deterministic order)."""
    n_batch, n_tail = per_batch.shape
    rc = load().reduce_axis0(_ptr(per_batch, "per_batch"), n_batch, n_tail,
                             _ptr(out, "out", (n_tail,)), _stream(stream))
    _check("reduce_axis0", rc)


def cfc_wait_self_test(stream=None) -> None:
    """Enqueue the self-test kernel whose bounded wait runs out (read the result with
    device_status(): 1 after about 2 s)."""
    _check("cfc_wait_self_test", load().cfc_wait_self_test(_stream(stream)))


def probe_fma(out, blocks: int, iters: int, stream=None) -> float:
    """Enqueue the fp32 FMA throughput probe; returns the flops it performs."""
    flop = ctypes.c_double(0)
    _check("cfc_probe_fma", load().cfc_probe_fma(_ptr(out, "out"), blocks, iters,
                                                 ctypes.byref(flop), _stream(stream)))
    return flop.value


def probe_l2_read(buf, passes: int, out, blocks: int, stream=None) -> float:
    """Enqueue the L2 read-bandwidth probe over ``buf``; returns the bytes it reads."""
    nbytes = ctypes.c_double(0)
    _check("cfc_probe_l2_read",
           load().cfc_probe_l2_read(_ptr(buf, "buf"), buf.numel(), passes, _ptr(out, "out"), blocks,
                                    ctypes.byref(nbytes), _stream(stream)))
    return nbytes.value


def copy(src, dst, stream=None) -> None:
    """dst <- src by the library's copy kernel.  Both are contiguous tensors of the same size in
    bytes (a multiple of 16, 16-byte aligned); each is on the device or in pinned host memory."""
    import torch

    for t, name in ((src, "src"), (dst, "dst")):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous torch.Tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or in pinned host memory")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst differ in size")
    _check("cfc_copy", load().cfc_copy(ctypes.c_void_p(src.data_ptr()),
                                       ctypes.c_void_p(dst.data_ptr()), nbytes, _stream(stream)))


def device_status() -> int:
    """Synchronise, then read and clear the device status word (0 = no kernel gave up)."""
    v = ctypes.c_int(0)
    _check("cfc_device_status", load().cfc_device_status(ctypes.byref(v)))
    return v.value


def forward_bf16_workspace_bytes(B: int, K: int, C: int, n_x: int) -> int:
    """Workspace of cfc_forward_bf16 (X = W_u u + b in fp32)."""
    out = ctypes.c_size_t(0)
    _check("cfc_forward_bf16_workspace_bytes",
           load().cfc_forward_bf16_workspace_bytes(B, K, C, n_x, ctypes.byref(out)))
    return out.value


def cfc_forward_bf16(u, h0, W, b, ts, H, cache, ws, stream=None) -> None:
    """bf16 H [K,B,C] and cache [K,B,3,C] <- the forward with fp32 arithmetic."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    wp, wn = _ws(ws)
    rc = load().cfc_forward_bf16(
        _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)), _ptr(W, "W", (4, C, n_in)),
        _ptr(b, "b", (4, C)), _ptr(ts, "ts", (K, B)), B, K, C, n_x,
        _ptr16(H, "H", (K, B, C)), _ptr16(cache, "cache", (K, B, 3, C)), wp, wn,
        _stream(stream))
    _check("cfc_forward_bf16", rc)


def cfc_backward_bf16(dH, u, h0, W, ts, H, cache, dW, db, du, dh0, ws, stream=None) -> None:
    """dW, db, du (optional), dh0 <- the backward of the bf16 H / cache of cfc_forward_bf16."""
    K, B, n_x = u.shape
    C = h0.shape[1]
    n_in = n_x + C
    wp, wn = _ws(ws)
    rc = load().cfc_backward_bf16(
        _ptr(dH, "dH", (K, B, C)), _ptr(u, "u", (K, B, n_x)), _ptr(h0, "h0", (B, C)),
        _ptr(W, "W", (4, C, n_in)), _ptr(ts, "ts", (K, B)), _ptr16(H, "H", (K, B, C)),
        _ptr16(cache, "cache", (K, B, 3, C)), B, K, C, n_x, _ptr(dW, "dW", (4, C, n_in)),
        _ptr(db, "db", (4, C)), _ptr(du, "du", (K, B, n_x)), _ptr(dh0, "dh0", (B, C)),
        wp, wn, _stream(stream))
    _check("cfc_backward_bf16", rc)


# ---- the pages' tau-decay cell ----

def decay_workspace_bytes(B: int, K: int, C: int, n_x: int) -> int:
    out = ctypes.c_size_t(0)
    _check("cfc_decay_workspace_bytes",
           load().cfc_decay_workspace_bytes(B, K, C, n_x, ctypes.byref(out)))
    return out.value


def cfc_decay_forward(x, h0, W, b, tau, ts, H, E, stream=None) -> None:
    """H [K,B,C] and E = tanh(a) [K,B,C] <- the tau-decay cell over K steps."""
    K, B, n_x = x.shape
    C = h0.shape[1]
    rc = load().cfc_decay_forward(
        _ptr(x, "x", (K, B, n_x)), _ptr(h0, "h0", (B, C)), _ptr(W, "W", (C, n_x + C)),
        _ptr(b, "b", (C,)), _ptr(tau, "tau", (C,)), _ptr(ts, "ts", (K, B)), B, K, C, n_x,
        _ptr(H, "H", (K, B, C)), _ptr(E, "E", (K, B, C)), _stream(stream))
    _check("cfc_decay_forward", rc)


def cfc_decay_backward(dH, x, h0, W, tau, ts, H, E, dW, db, dtau, dx, dh0, ws,
                       stream=None) -> None:
    """dW, db, dtau, dx (optional), dh0 <- BPTT of the tau-decay cell."""
    K, B, n_x = x.shape
    C = h0.shape[1]
    wp, wn = _ws(ws)
    rc = load().cfc_decay_backward(
        _ptr(dH, "dH", (K, B, C)), _ptr(x, "x", (K, B, n_x)), _ptr(h0, "h0", (B, C)),
        _ptr(W, "W", (C, n_x + C)), _ptr(tau, "tau", (C,)), _ptr(ts, "ts", (K, B)),
        _ptr(H, "H", (K, B, C)), _ptr(E, "E", (K, B, C)), B, K, C, n_x,
        _ptr(dW, "dW", (C, n_x + C)), _ptr(db, "db", (C,)), _ptr(dtau, "dtau", (C,)),
        _ptr(dx, "dx", (K, B, n_x)), _ptr(dh0, "dh0", (B, C)), wp, wn, _stream(stream))
    _check("cfc_decay_backward", rc)
