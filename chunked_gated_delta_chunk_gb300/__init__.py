"""chunked_gated_delta_chunk_gb300 — chunked Gated DeltaNet prefill for GB300.

The compute path is the CUDA library ``libgdn.so`` (sm_103a kernels behind a
C ABI declared in ``include/gdn.h``).  ``binding`` is a thin ctypes layer over
it with the same entry-point names; ``build`` compiles it in-tree.  Importing
this package loads nothing: the library is loaded on first use of
``binding`` and a missing library is an error, never a fallback.
"""

__all__ = ["binding", "build", "inputs"]
