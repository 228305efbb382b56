"""cfc_copy, the copy kernel that moves a step's inputs in from pinned host memory and its
gradients back out: byte-exact in both directions at ragged sizes, and refusing memory the
device cannot reach or overlapping ranges without launching anything."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

INVALID_ARG = -8


@pytest.mark.parametrize("nbytes", [16, 48, 4096, 65536 + 16, 1 << 20, (7 << 20) + 48])
def test_copy_round_trip_is_exact(nbytes):
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    _lib.copy(src, dev)
    _lib.copy(dev, back)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)
    # device to device as well, in a graph
    dev2 = torch.empty_like(dev)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        _lib.copy(dev, dev2)
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(dev2, dev)
    assert _lib.device_status() == 0


def test_copy_refuses_unreachable_or_overlapping_memory():
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    lib = _lib.load()
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pageable = np.zeros(4096 + 16, dtype=np.uint8)
    off = (-pageable.ctypes.data) % 16
    host = ctypes.c_void_p(pageable.ctypes.data + off)  # never registered with CUDA
    d = ctypes.c_void_p(dev.data_ptr())
    assert lib.cfc_copy(host, d, 4096, None) == INVALID_ARG
    assert lib.cfc_copy(d, host, 4096, None) == INVALID_ARG
    assert lib.cfc_copy(d, ctypes.c_void_p(dev.data_ptr() + 1024), 2048, None) == INVALID_ARG
    torch.cuda.synchronize()
    assert int(dev.sum()) == 0
