"""prefix_cached_kv_radix_gb300: prefix-cached KV attention with a radix tree on GB300.

The compute lives in libradixattn.so (include/radix_attn.h): a host C++ radix tree with
LRU eviction over KV-pool slots, and sm_103a kernels for the slot table / K-V scatter,
extend attention (tcgen05 + TMEM) and split-KV decode attention.  ``api`` is the thin
ctypes binding; ``engine`` strings the calls into one prefix-cached step; ``build``
compiles the library in-tree.
"""
from . import api  # noqa: F401
