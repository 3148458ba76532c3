"""Packed varlen (document-masked) attention for one GB300 (sm_103a).

The compute path is the C-ABI library ``libpva.so`` (include/pva.h); this
package holds the thin ctypes binding (``api``), the build step
(``build``) and the seeded synthetic workloads (``workloads``).  Importing
the package does not load the library; the first call does, and fails
loudly if it has not been built.
"""
from .workloads import (MASK_CAUSAL, MASK_SHARED_QUESTION, MASK_SLICES, MASK_SLIDING_WINDOW,
                        MASK_ZIGZAG_PAIR)

__all__ = ["MASK_CAUSAL", "MASK_SLIDING_WINDOW", "MASK_SHARED_QUESTION", "MASK_ZIGZAG_PAIR",
           "MASK_SLICES"]
