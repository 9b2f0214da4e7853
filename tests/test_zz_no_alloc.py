"""pkv_paged_attn_decode_noalloc, the decode entry point for callers that
cannot allocate device memory (an engine that owns all of HBM through its own
KV block pool, or a decode path where cudaMalloc's device-wide sync is not
acceptable).  It keeps the split-KV partials in a fixed array inside the
library, so the caller passes only inputs and outputs.

Called through the C ABI and checked against the regular entry point (which
takes a caller-allocated workspace) within the parity tolerance, and against
the oracle, on calls in a row so that each call runs over the previous call's
leftover scratch; the mma.sync, CUDA-core and tcgen05 kernels all go through
it.  This file is collected last on purpose (conftest.py also moves it to the
end of the run), so a run that stops at its first failure has run every
other test first."""
from __future__ import annotations

import ctypes

import pytest
import torch

from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, oracle_decode, widen_out

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.pkv_paged_attn_decode_noalloc
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _call_noalloc(pkv, d, out, scale, max_context_len, split_tokens=0, kernel=0):
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], max_context_len,
                             split_tokens, kernel)
    f = _noalloc(pkv.load_library())
    return f(ctypes.addressof(shape), d["q"].data_ptr(), d["k_cache"].data_ptr(),
             d["v_cache"].data_ptr(), d["block_tables"].data_ptr(),
             d["context_lens"].data_ptr(), scale, out.data_ptr(),
             torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point(pkv):
    cases = [  # (batch, kernel): calls in a row, different batches and kernels
        (W.make(W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 3000, lens="fixed"), seed=1), 0),
        (W.make(W.scaled(W.WORKLOADS["llama7b_mha"], 6, 1300), seed=2), 0),
        (W.make(W.scaled(W.WORKLOADS["llama3_8b_gqa"], 8, 1500, min_len=16), seed=3), 3),
        (W.make(W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 3000, lens="fixed"), seed=4), 3),
    ]
    for w, kernel in cases:
        d = device_inputs(w)
        shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len,
                                 0, kernel)
        assert pkv.decode_plan(shape).workspace_bytes > 0  # the scratch is really used
        out = torch.full_like(d["q"], float("nan"))
        assert _call_noalloc(pkv, d, out, w.scale, w.max_context_len, kernel=kernel) == 0
        ref = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], w.scale,
                                    max_context_len=w.max_context_len, kernel=kernel)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        name = f"{w.spec.name} kernel={kernel}"
        assert_close(widen_out(out), widen_out(ref), f"noalloc vs workspace, {name}")
        assert_close(widen_out(out), oracle_decode(w), f"noalloc vs oracle, {name}")


def test_noalloc_rejects_oversized_partials(pkv):
    # 256 sequences x 64 heads x 2048 partitions of 16 tokens: far beyond
    # 64 MiB of partials, rejected on the host before anything is enqueued
    spec = W.WorkloadSpec("big", 256, 64, 8, 128, 16, W.BF16, 300, 2048, "fixed", (1,) * 256)
    w = W.make(spec, seed=0)
    d = device_inputs(w)
    out = torch.empty_like(d["q"])
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], 2048 * 16, 16)
    assert pkv.decode_plan(shape).workspace_bytes > 64 << 20
    n0 = pkv.launch_count()
    assert _call_noalloc(pkv, d, out, w.scale, 2048 * 16, split_tokens=16) == -5
    assert pkv.launch_count() == n0
