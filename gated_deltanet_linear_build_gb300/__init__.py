"""GDN token-mixer hot path for GB300 (sm_103a).

The compute lives in ``libgdn_gb300.so`` (C ABI in ``include/gdn.h``);
``gdn`` is its ctypes binding, ``synth`` the seeded input generators and
``build`` the nvcc build step.
"""
from . import build  # noqa: F401
