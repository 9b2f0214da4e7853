"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding and the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W

# |gpu - ref| <= ATOL + RTOL * |ref|, elementwise (fp16/bf16 output, fp32 accumulate)
ATOL, RTOL = 2e-3, 1e-2


def widen_out(out: torch.Tensor) -> np.ndarray:
    return out.detach().to(torch.float64).cpu().numpy()


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite outputs"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={gpu[i]} ref={ref[i]} err={err[i]:.3g}")


def device_inputs(w: W.Workload):
    dev = torch.device("cuda")
    return dict(q=w.q.to(dev), k_cache=w.k_cache.to(dev), v_cache=w.v_cache.to(dev),
                block_tables=torch.from_numpy(w.block_tables).to(dev),
                context_lens=torch.from_numpy(w.context_lens).to(dev))


def gpu_decode(pkv, w: W.Workload, d=None, split_tokens: int = 0, max_context_len=None):
    d = d or device_inputs(w)
    out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], w.scale, split_tokens=split_tokens,
                                max_context_len=max_context_len or w.max_context_len)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return out


def oracle_decode(w: W.Workload, k_cache=None, v_cache=None):
    return oracle.decode(W.bits(w.q), W.bits(w.k_cache if k_cache is None else k_cache),
                         W.bits(w.v_cache if v_cache is None else v_cache), w.block_tables,
                         w.context_lens, w.scale, w.spec.dtype)
