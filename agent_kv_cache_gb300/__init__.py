"""Active-KV cache operations for agent serving on GB300 (sm_103a).

The compute lives in the CUDA library ``libakv.so`` (include/akv.h); this
package builds it (:func:`build`), binds it with ctypes (:mod:`.abi`, the same
names as the C ABI) and offers :class:`Cache`, a small owner of the two
device pools (allocated with PyTorch, which is only used for device memory
and streams).
"""
from ._build import build, LIB as LIB_PATH
from . import abi
from .cache import Cache, PrefixIndex

__all__ = ["build", "LIB_PATH", "abi", "Cache", "PrefixIndex"]
