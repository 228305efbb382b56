"""GB300 (sm_103a) CfC K-loop: forward recurrence, BPTT and deterministic gradients.

The compute lives in libcfc.so (C ABI in include/cfc.h, kernels in csrc/); this package holds
its ctypes binding (``_lib``), the step object (``step.KLoopStep``), the seeded synthetic
inputs (``inputs``) and the build script (``build``).
"""
from .inputs import CONFIGS, Workload, custom, make_inputs  # noqa: F401
