"""Properties of the CUDA path that hold at any size: bitwise determinism, graph replay equal to
eager, overwrite semantics (a second call reflects only its own inputs), the batch gradient
equals the sum of single-row gradients, and reduce_axis0 against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_helpers import GRAD_TOL, outputs_np, run_gpu
from recurrent_cfc_cell_gb300 import inputs

pytestmark = pytest.mark.gpu

KEYS = ("H", "cache", "d_pre", "dW", "db", "du", "dh0")


def _step(w):
    import torch

    from recurrent_cfc_cell_gb300 import build
    from recurrent_cfc_cell_gb300.step import KLoopStep, to_device

    build.build()
    inp = inputs.make_inputs(w)
    st = KLoopStep(w.B, w.K, w.C, w.n_x).bind(**to_device(inp))
    return st, inp, torch


DETERMINISM_CASES = [
    inputs.CONFIGS[1],                                  # contractions split together, paired merge
    inputs.CONFIGS[3],                                  # dW split over 128 CTAs, du unsplit
    inputs.custom(B=1030, K=6, n_x=16, C=256, seed=8),  # cluster-split tensor-core BPTT
]


@pytest.mark.parametrize("w", DETERMINISM_CASES, ids=lambda w: w.name)
def test_bitwise_deterministic_runs(w):
    st, _, torch = _step(w)
    st.run()
    torch.cuda.synchronize()
    first = {k: v.clone() for k, v in st.outputs().items()}
    for _ in range(3):
        st.run()
        torch.cuda.synchronize()
        for k, v in st.outputs().items():
            assert torch.equal(v, first[k]), k


def test_graph_replay_bitwise_equals_eager():
    st, _, torch = _step(inputs.CONFIGS[1])
    st.run()
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in st.outputs().items()}
    for k, v in st.outputs().items():
        v.fill_(float("nan") if v.is_floating_point() else -1)
    st.capture()
    st.replay()
    torch.cuda.synchronize()
    for k, v in st.outputs().items():
        assert torch.equal(v, eager[k]), k


def test_second_call_reflects_only_its_inputs():
    """Successor of the spec's cfc_bwd_scratch_clears_between_steps: step B after step A must
    equal step B alone (no output or scratch carries anything over)."""
    import torch

    from recurrent_cfc_cell_gb300.step import to_device

    st, inp_a, _ = _step(inputs.CONFIGS[1])
    w = inputs.CONFIGS[1]
    inp_b = inputs.make_inputs(inputs.Workload(w.name, w.B, w.K, w.n_x, w.C, seed=99))
    st.run()
    st.bind(**to_device(inp_b))
    st.run()
    torch.cuda.synchronize()
    after_a = outputs_np(st)
    fresh = run_gpu(inp_b)
    for k in KEYS:
        assert np.array_equal(after_a[k], fresh[k]), k


def test_batch_gradient_is_sum_of_single_row_gradients():
    """Successor of the spec's cfc_bwd_b1_matches_single_sample: run each row alone (B=1) and
    check the batch's dW, db equal the sum and H, du, dh0 match per row."""
    w = inputs.custom(B=6, K=9, n_x=12, C=64, seed=5)
    inp = inputs.make_inputs(w)
    full = run_gpu(inp)
    acc_dW = np.zeros_like(full["dW"], dtype=np.float64)
    acc_db = np.zeros_like(full["db"], dtype=np.float64)
    for b in range(w.B):
        one = {"u": np.ascontiguousarray(inp["u"][:, b:b + 1]),
               "h0": np.ascontiguousarray(inp["h0"][b:b + 1]), "W": inp["W"], "b": inp["b"],
               "ts": np.ascontiguousarray(inp["ts"][:, b:b + 1]),
               "dH": np.ascontiguousarray(inp["dH"][:, b:b + 1])}
        o = run_gpu(one)
        acc_dW += o["dW"]
        acc_db += o["db"]
        assert np.array_equal(o["H"][:, 0], full["H"][:, b])
        assert oracle.rel_err(o["du"][:, 0], full["du"][:, b]) <= 1e-6
        assert oracle.rel_err(o["dh0"][0], full["dh0"][b]) <= 1e-6
    assert oracle.rel_err(full["dW"], acc_dW) <= GRAD_TOL
    assert oracle.rel_err(full["db"], acc_db) <= GRAD_TOL


def test_device_status_clean_after_runs():
    from recurrent_cfc_cell_gb300 import _lib

    run_gpu(inputs.make_inputs(inputs.CONFIGS[0]))
    assert _lib.device_status() == 0


@pytest.mark.parametrize("n_batch,n_tail,offset", [(1, 1, 0), (37, 11, 0), (2048, 512, 0),
                                                   (16, 1407, 0), (300, 64, 1), (5000, 96, 0),
                                                   (20000, 1024, 0)])
def test_reduce_axis0(n_batch, n_tail, offset):
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    rng = np.random.default_rng(n_batch * 31 + n_tail)
    a = rng.normal(0, 1, size=(n_batch, n_tail)).astype(np.float32)
    flat = torch.empty(a.size + offset, dtype=torch.float32, device="cuda")
    dev = flat[offset:].view(n_batch, n_tail)  # offset 1 -> 4-byte aligned, scalar path
    dev.copy_(torch.from_numpy(a))
    out = torch.full((n_tail,), float("nan"), device="cuda")
    _lib.reduce_axis0(dev, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.reduce_axis0(a)
    scale = np.sqrt(n_batch) * 1e-6 * max(1.0, np.log2(n_batch))
    assert np.max(np.abs(got - ref)) <= scale * max(1.0, np.max(np.abs(a))) * 4
    out2 = torch.full((n_tail,), 123.0, device="cuda")
    _lib.reduce_axis0(dev, out2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)  # bitwise reproducible, fully overwritten


def test_reduce_axis0_vector_and_scalar_paths_agree_bitwise():
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    rng = np.random.default_rng(3)
    a = torch.from_numpy(rng.normal(0, 1, size=(999, 256)).astype(np.float32)).cuda()
    flat = torch.empty(a.numel() + 1, device="cuda")
    shifted = flat[1:].view(999, 256)
    shifted.copy_(a)
    o1 = torch.empty(256, device="cuda")
    o2 = torch.empty(256, device="cuda")
    _lib.reduce_axis0(a, o1)
    _lib.reduce_axis0(shifted, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
