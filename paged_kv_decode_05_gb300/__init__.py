"""pkv: paged-KV decode attention for one GB300 (sm_103a).

The product is the C-ABI library ``libpkv.so`` (kernels in ``csrc/``,
declarations in ``include/pkv.h``). ``binding`` is a thin ctypes layer with the
same entry-point names that marshals torch CUDA tensors into plain pointers.
Importing this package loads nothing; the library is loaded on first use and a
missing or stale build raises instead of falling back to anything else.
"""

__all__ = ["binding", "workloads", "build"]
