"""GB300-native paged K/V-cache decode path (PagedAttention's data-parallel hot path).

* ``binding``   -- ctypes binding of libpkv.so (include/pkv.h): paged decode
                   attention, reshape_and_cache, copy_blocks, host block manager.
* ``workloads`` -- seeded synthetic inputs (no method arithmetic).
* ``_build``    -- in-tree nvcc build of libpkv.so for sm_103a.

Importing the package loads nothing; ``binding.load()`` (called by every
binding function) loads the library and raises if it was not built.
"""

__all__ = ["binding", "workloads"]
