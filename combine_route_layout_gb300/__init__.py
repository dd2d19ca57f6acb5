"""GB300-native MoE expert-parallel dispatch / combine (simulated EP ranks on one GPU).

The compute lives in libep.so (hand-written sm_103a CUDA kernels behind the C
ABI of include/ep.h); `ep` is its thin Python binding.
"""
from . import ep  # noqa: F401
from .ep import EpDispatchCombineConfig, EpDispatchCombineOp, EpError  # noqa: F401
