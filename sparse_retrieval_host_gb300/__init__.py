"""GB300-native FlashMemory LSA + KV_SWAP decode-step hot path.

The compute runs in libsrh.so (hand-written sm_103a CUDA kernels behind the C
ABI of include/srh.h); this package is its ctypes binding (``abi``), a thin
buffer/stream helper (``runtime``) and the build script (``build``).
"""
from . import abi  # noqa: F401

__all__ = ["abi"]
