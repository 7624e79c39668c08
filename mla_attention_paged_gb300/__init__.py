"""GB300-native MLA attention over a paged latent KV cache.

The compute path is the C-ABI library ``libmla.so`` (hand-written CUDA for sm_103a,
declared in ``include/mla.h``); ``mla_attention_paged_gb300.mla`` is its thin ctypes
binding.  Importing this package loads nothing; import ``.mla`` to use the library.
"""
__all__ = ["mla", "inputs"]
