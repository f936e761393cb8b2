"""Group-32 low-bit (4-bit asymmetric / 2-bit Lloyd-Max codebook) weight-only
decode GEMV for GB300 (sm_103a).

The compute lives in ``_lib/liblbq.so`` (C ABI in ``include/lbq.h``);
``lbq`` is its thin binding and ``synth`` the seeded input generators.
Importing the package loads nothing; the library is loaded on first use and
raises ImportError if it has not been built.
"""

__all__ = ["lbq", "synth"]
