"""GB300-native batched paged-attention decode read and KV append.

The compute path is the C-ABI library ``libnsv.so`` (hand-written CUDA for
sm_103a, sources in ``csrc/``, declarations in ``include/nsv.h``).  The thin
ctypes binding is ``paged_kv_decode_nsv_gb300.nsv``; importing it loads the
library and raises if the library has not been built.  ``workloads`` builds
seeded synthetic batches and holds none of the read's arithmetic.
"""

__all__ = ["nsv", "workloads"]
