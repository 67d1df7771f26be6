"""Collective KV cache path for GB300 (sm_103a): the data-parallel core of TokenDance's
collective KV cache sharing for multi-agent All-Gather rounds.

`collective_kv_cache_gb300.td` is the thin ctypes binding of the C-ABI library
(include/td.h); `collective_kv_cache_gb300.synth` draws seeded synthetic rounds.
"""
