"""Exact IO-aware attention for NVIDIA GB300 (sm_103a).

The computation runs in libfa.so (hand-written CUDA, C ABI in include/fa.h);
this package is its Python binding plus the seeded input generators.
"""
from .binding import (FAError, attention, backward, backward_workspace_bytes, default_num_splits,
                      device_status, forward, load_library, measure_exp2_rate, profile_collect,
                      profile_enable)

__all__ = ["FAError", "attention", "backward", "backward_workspace_bytes", "default_num_splits",
           "device_status", "forward", "load_library", "measure_exp2_rate", "profile_collect",
           "profile_enable"]
