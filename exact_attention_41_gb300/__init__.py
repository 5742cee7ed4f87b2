"""libattn for GB300 (sm_103a): exact scaled dot-product attention.

The compute path lives in the CUDA library ``libattn.so`` (sources under
``csrc/``, C ABI in ``include/libattn.h``); ``exact_attention_41_gb300.libattn``
is the thin ctypes binding over it.  Importing this package does not load the
library; the binding loads it on first use and raises if it is missing.
"""
__all__ = ["libattn", "synthetic"]
