"""Hybrid local/global grouped-query attention for B300 (sm_103a).

The compute path is ``libmg.so`` (hand-written CUDA, C ABI declared in
``include/mg.h``); ``hybrid_local_global_attn_b300.mg`` is its thin ctypes
binding.  Importing this package loads nothing; importing ``.mg`` loads the
library and fails loudly if it has not been built.
"""
__all__ = ["mg", "synth"]
