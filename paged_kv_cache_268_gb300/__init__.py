"""Paged KV-cache decode attention for GB300 (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA behind a C ABI, see
``include/pkv.h``); this package is a thin ctypes binding over it plus the
seeded workload generator used by the tests and the benchmark.
"""
