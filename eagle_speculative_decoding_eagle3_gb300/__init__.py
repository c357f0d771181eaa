"""GB300-native (sm_103a) EAGLE-3 draft head for an MLA (DeepseekV3-shaped) target.

The compute lives in libeagle3.so (CUDA kernels behind the C ABI in include/eagle3.h);
``eagle3`` is its ctypes binding and ``harness`` moves seeded workloads into HBM.
"""
from . import eagle3  # noqa: F401
