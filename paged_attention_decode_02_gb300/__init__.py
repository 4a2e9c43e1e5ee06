"""Paged-attention decode for GB300 (sm_103a).

The compute path lives in ``libpa_decode.so`` (hand-written CUDA behind a C ABI,
see ``include/pa_decode.h``).  ``ops`` is the thin ctypes binding; ``synth``
makes seeded synthetic workloads.  Importing the package loads nothing: the
shared library is opened on first use, and a missing library is an error.
"""

__all__ = ["ops", "synth"]
