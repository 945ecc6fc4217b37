"""GB300-native (sm_103a) Megatron tensor-parallel transformer layer.

The layer runs in the CUDA library libmtl.so (C ABI: include/mtl.h); the
`mtl` module is its ctypes binding.
"""
from . import mtl  # noqa: F401
