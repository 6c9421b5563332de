"""GB300-native BN254 G1 multi-scalar multiplication.

``MsmG1`` wraps the C ABI of ``libmsm_g1.so`` (include/msm_g1.h); the kernels
live in ``csrc/``.  ``synth`` draws seeded synthetic workloads.
"""
from .msm import MsmG1, MsmError, lib, to_device, to_host  # noqa: F401
