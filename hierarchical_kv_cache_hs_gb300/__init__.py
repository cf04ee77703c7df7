"""HiSparse swap-in path on GB300: top-k resolve against a per-request hot
device buffer backed by a pinned host KV pool.

Importing the package loads nothing native.  ``hierarchical_kv_cache_hs_gb300.hs``
is the binding to the CUDA library (it raises if the library is not built);
``hierarchical_kv_cache_hs_gb300.tracegen`` produces the seeded synthetic inputs.
"""
