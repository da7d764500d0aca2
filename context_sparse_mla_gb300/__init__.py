"""GB300-native context-parallel (PCP) prefill attention over MLA latent KV.

The compute path lives in ``libcpmla.so`` (hand-written sm_103a CUDA behind a C
ABI, headers in ``include/cpmla.h``).  ``cpmla`` is the thin ctypes binding with
the same entry-point names; ``synth`` draws seeded synthetic inputs.  Importing
the package loads nothing: the library is opened on first use and a missing
library is an error, never a fallback.
"""
__all__ = ["cpmla", "synth"]
