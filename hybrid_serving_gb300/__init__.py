"""GB300-native exact tree-structured prefill (ForkAttention + Gated DeltaNet
fork prefill) behind the C ABI of include/hs.h.

The compute runs in libhsfork.so (CUDA for sm_103a); this package holds the
library sources (``csrc/``), its build (``_build``), the ctypes binding
(``_lib``) and thin Python wrappers (``api``, ``rounds``).  Importing
``api`` fails loudly when the library is not built -- there is no fallback.
"""
__all__ = ["api", "rounds"]
