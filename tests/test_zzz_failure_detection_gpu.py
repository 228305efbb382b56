"""Failure detection on the device without a fault: a kernel's bounded wait on an mbarrier
that nothing completes runs out, the status word reports it, and the context stays usable.
(Named to run after the other GPU tests: while the self-test kernel waits, no other kernel of
the library should be running.)"""
import time

import pytest

from gpu_helpers import assert_parity, oracle_ref, run_gpu
from recurrent_cfc_cell_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_abandoned_wait_is_reported_and_the_context_stays_usable():
    import torch

    from recurrent_cfc_cell_gb300 import _lib, build

    build.build()
    assert _lib.device_status() == 0
    t0 = time.perf_counter()
    _lib.cfc_wait_self_test()
    status = _lib.device_status()  # synchronises
    dt = time.perf_counter() - t0
    assert status == 1
    assert 1.9 < dt < 60.0, dt
    assert _lib.device_status() == 0  # read and cleared
    # the device still runs a step correctly
    inp = inputs.make_inputs(inputs.custom(B=5, K=7, n_x=5, C=40, seed=41))
    assert_parity(run_gpu(inp), oracle_ref(inp))
    torch.cuda.synchronize()
    assert _lib.device_status() == 0
