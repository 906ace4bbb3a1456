"""B300-native (sm_103a) forward pass of one Mixture-of-Experts FFN layer.

The computation lives in libmoe.so (CUDA kernels behind the C ABI of
include/moe.h); this package is its ctypes binding. Importing it does not load
the library; the first call does, and fails loudly if it has not been built.
"""
from .binding import *  # noqa: F401,F403
from .binding import EXPORTS, MoeConfig, MoeError, MoeRoutingStats, lib, make_config, alloc_workspace  # noqa: F401
