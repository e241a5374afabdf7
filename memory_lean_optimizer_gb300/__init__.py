"""GB300-native fused optimizer-step engine for memory-lean full fine-tuning.

The compute path is liblmopt.so (CUDA kernels for sm_103a behind the C ABI of include/lmopt.h).
``lmopt`` is its ctypes binding; ``engine`` holds the torch-facing group objects (PyTorch only
provides device memory and streams); ``workloads`` holds the seeded synthetic workloads.
"""
from . import lmopt  # noqa: F401

__all__ = ["lmopt"]
