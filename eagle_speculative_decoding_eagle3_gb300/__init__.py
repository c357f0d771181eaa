"""GB300-native (sm_103a) EAGLE-3 draft heads for an MLA (DeepseekV3-shaped) target: the MLA draft
head and the Llama-style MHA draft head, with bf16 / fp32, FP8 E4M3 or NVFP4 projection weights.

The compute lives in libeagle3.so (CUDA kernels behind the C ABI in include/eagle3.h);
``eagle3`` is its ctypes binding and ``harness`` moves seeded workloads into HBM.
"""
from . import eagle3  # noqa: F401
