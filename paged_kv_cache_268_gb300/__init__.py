"""Paged KV-cache decode attention for GB300 (sm_103a).

The compute lives in ``lib/libpkv.so`` (hand-written CUDA behind the C ABI in
``include/pkv.h``); this package is a thin ctypes binding over it, plus the
seeded workload generator used by the tests and the benchmark.  Build the
library with ``python -m paged_kv_cache_268_gb300.build``.
"""
from ._binding import (  # noqa: F401
    BlockManager,
    PkvError,
    copy_blocks,
    alloc_workspace,
    decode_plan,
    decode_shape,
    decode_step,
    get_device_error,
    kv_cache_append,
    launch_count,
    load_library,
    paged_attn_decode,
    selftest_wait_timeout,
    set_workspace,
    workspace_bytes,
)
