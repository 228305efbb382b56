"""cfc_backward_noalloc: the backward pass for callers that cannot allocate device memory (a
plugin hosted by a framework that owns the GPU's memory, a program with a fixed device memory
footprint).  It must give the same results as cfc_backward with a caller-allocated workspace,
call after call, although every call reuses the one scratch array built into the library.

Kept in a file of its own that pytest collects last, so a run that stops at its first failure
has already run every other test.  It also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import GRAD_TOL
from recurrent_cfc_cell_gb300 import inputs

pytestmark = pytest.mark.gpu

OUT = ("dW", "db", "du", "dh0")


def _setup(w, mode, with_du):
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build
    from recurrent_cfc_cell_gb300.step import KLoopStep, to_device

    build.build()
    lib = _lib.load()
    d = to_device(inputs.make_inputs(w))
    st = KLoopStep(w.B, w.K, w.C, w.n_x, dw_mode=mode, with_du=with_du).bind(**d)
    st.forward()
    return lib, st, d, torch


def _noalloc(lib, st, d, torch):
    """Call cfc_backward_noalloc through the C ABI into fresh (NaN-filled) output tensors."""
    f32 = dict(dtype=torch.float32, device=st.device)
    out = {"dW": torch.full((4, st.C, st.n_in), float("nan"), **f32),
           "db": torch.full((4, st.C), float("nan"), **f32),
           "dh0": torch.full((st.B, st.C), float("nan"), **f32)}
    if st.du is not None:
        out["du"] = torch.full((st.K, st.B, st.n_x), float("nan"), **f32)

    def p(t):
        return ctypes.c_void_p(t.data_ptr()) if t is not None else None

    rc = lib.cfc_backward_noalloc(
        p(d["dH"]), p(d["u"]), p(d["h0"]), p(d["W"]), p(d["ts"]), p(st.H), p(st.cache),
        st.B, st.K, st.C, st.n_x, p(out["dW"]), p(out["db"]), p(out.get("du")), p(out["dh0"]),
        st.dw_mode, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.cfc_error_string(rc)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _reference(st, torch):
    """The existing entry point, with a workspace allocated by the caller."""
    st.backward()
    torch.cuda.synchronize()
    return {k: getattr(st, k).cpu().numpy() for k in OUT if getattr(st, k) is not None}


def _rel(x, y):
    den = max(float(np.max(np.abs(y))), 2.0 ** -126)
    return float(np.max(np.abs(x - y))) / den


CASES = [
    (inputs.CONFIGS[1], 0, True),                               # the pages' shape
    (inputs.custom(B=5, K=7, n_x=5, C=40, seed=4), 0, True),    # ragged sizes
    (inputs.CONFIGS[2], 0, True),                               # 32 x 64 x 256 fits too
    (inputs.CONFIGS[1], 3, True),                               # CUDA-core contraction
    (inputs.CONFIGS[1], 0, False),                              # du not requested
]


@pytest.mark.parametrize("w,mode,with_du", CASES,
                         ids=[f"{w.name}-mode{m}-{'du' if du else 'nodu'}" for w, m, du in CASES])
def test_noalloc_matches_backward_on_two_calls(w, mode, with_du):
    lib, st, d, torch = _setup(w, mode, with_du)
    from recurrent_cfc_cell_gb300 import _lib

    assert _lib.workspace_bytes(w.B, w.K, w.C, w.n_x, mode) <= _lib.NOALLOC_SCRATCH_BYTES
    # Two calls in a row: the second reuses the scratch the first one left behind.
    for call in range(2):
        if call == 1:  # a new upstream gradient, so anything stale in the scratch would show
            d["dH"].mul_(-0.5).add_(0.25)
        got = _noalloc(lib, st, d, torch)
        ref = _reference(st, torch)
        assert set(got) == set(ref)
        for k in got:
            assert np.all(np.isfinite(got[k])), (call, k)
            assert _rel(got[k], ref[k]) <= GRAD_TOL, (call, k, _rel(got[k], ref[k]))


def test_noalloc_rejects_problems_beyond_its_scratch():
    from recurrent_cfc_cell_gb300 import _lib

    lib = _lib.load()
    w = inputs.CONFIGS[3]  # B=256, K=64, C=128: its d_pre alone is 32 MiB
    assert _lib.workspace_bytes(w.B, w.K, w.C, w.n_x) > _lib.NOALLOC_SCRATCH_BYTES
    f = ctypes.c_void_p(0x10000)
    rc = lib.cfc_backward_noalloc(*([f] * 7), w.B, w.K, w.C, w.n_x, *([f] * 4), 0, None)
    assert rc == _lib.CFC_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.cfc_error_string(rc)
