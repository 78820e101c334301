"""GB300-native paged KV-cache decode: one block pool, block tables, and
hand-written sm_103a kernels behind the C ABI in ``include/pagedattn.h``.

Submodules (import them explicitly):
  ``binding``    ctypes marshalling of every C entry point (same names).
  ``pool``       ``BlockPool``: torch-owned pool tensor + library handle.
  ``workloads``  seeded synthetic workloads shaped like the source pages' examples.

The CUDA library is loaded on first use of ``binding``; that fails loudly when
the library has not been built.
"""
