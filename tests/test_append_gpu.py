"""GPU parity of kv_cache_append against the oracle: bit-exact over the whole
cache (untouched slots, including NaN-poisoned ones, must not change)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, gpu_decode, oracle_decode, widen_out
from test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu


def _append_and_compare(pkv, w: W.Workload, slots: np.ndarray, k_new=None, v_new=None):
    k_new = w.k_new if k_new is None else k_new
    v_new = w.v_new if v_new is None else v_new
    kc, vc = w.k_cache.cuda().clone(), w.v_cache.cuda().clone()
    before_k, before_v = W.bits(kc), W.bits(vc)
    pkv.kv_cache_append(k_new.cuda(), v_new.cuda(), torch.from_numpy(slots).cuda(), kc, vc)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    ek, ev = oracle.append(W.bits(k_new), W.bits(v_new), slots, before_k, before_v)
    assert np.array_equal(W.bits(kc), ek)
    assert np.array_equal(W.bits(vc), ev)
    return kc, vc


@pytest.mark.parametrize("name", W.ORDER)
def test_append_small(pkv, name):
    w = W.make(SMALL[name], seed=1)
    slots = w.slot_mapping.copy()
    slots[::3] = -1                      # padding tokens write nothing
    _append_and_compare(pkv, w, slots)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_many_tokens(pkv, D):
    """A prefill-sized scatter: many tokens per call, random distinct slots."""
    spec = W.WorkloadSpec("append", 1, 4, 4, D, 16, W.BF16, 300, 300, "fixed", (4000,))
    w = W.make(spec, seed=D)
    rng = np.random.default_rng(D)
    T = 1500
    slots = rng.choice(spec.num_blocks * spec.block_size, size=T, replace=False).astype(np.int32)
    slots[rng.random(T) < 0.1] = -1
    g = torch.Generator().manual_seed(D)
    k_new = torch.randn((T, 4, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, 4, D), generator=g).to(torch.bfloat16)
    _append_and_compare(pkv, w, slots, k_new, v_new)


def test_append_bad_slot_sets_device_error(pkv):
    w = W.make(SMALL["llama7b_mha"], seed=0)
    slots = w.slot_mapping.copy()
    slots[0] = w.spec.num_blocks * w.spec.block_size          # one past the pool
    kc, vc = w.k_cache.cuda().clone(), w.v_cache.cuda().clone()
    before = W.bits(kc)
    pkv.kv_cache_append(w.k_new.cuda(), w.v_new.cuda(), torch.from_numpy(slots).cuda(), kc, vc)
    assert pkv.get_device_error() == 3
    slots[0] = -1
    ek, _ = oracle.append(W.bits(w.k_new), W.bits(w.v_new), slots, before, W.bits(w.v_cache))
    assert np.array_equal(W.bits(kc), ek)     # the bad row was skipped, the rest landed


def test_append_then_decode_small(pkv):
    """Continuous-batching step: append one token per sequence, then decode
    over lengths that include it; the oracle does the same on the host."""
    w = W.make(SMALL["cont_batch"], seed=4)
    d = device_inputs(w)
    pkv.kv_cache_append(w.k_new.cuda(), w.v_new.cuda(), torch.from_numpy(w.slot_mapping).cuda(),
                        d["k_cache"], d["v_cache"])
    out = gpu_decode(pkv, w, d)
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                           W.bits(w.k_cache), W.bits(w.v_cache))
    assert_close(widen_out(out), oracle_decode(w, ek, ev), "append+decode")


def test_append_then_decode_full_cont_batch(pkv):
    """The full continuous-batching workload (256 sequences, shared 512-token
    prefixes): bit-exact caches after the append, sampled decode rows."""
    w = W.make("cont_batch", seed=0, device="cuda")
    d = device_inputs(w)
    before_k, before_v = W.bits(d["k_cache"]), W.bits(d["v_cache"])
    pkv.kv_cache_append(w.k_new, w.v_new, torch.from_numpy(w.slot_mapping).cuda(),
                        d["k_cache"], d["v_cache"])
    out = widen_out(gpu_decode(pkv, w, d))
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping, before_k, before_v)
    assert np.array_equal(W.bits(d["k_cache"]), ek) and np.array_equal(W.bits(d["v_cache"]), ev)
    rng = np.random.default_rng(1)
    rows = np.array([(i, int(rng.integers(32))) for i in range(0, 256, 5)], dtype=np.int32)
    ref = oracle.decode_rows(rows, W.bits(w.q), ek, ev, w.block_tables, w.context_lens,
                             w.scale, w.spec.dtype)
    assert_close(out[rows[:, 0], rows[:, 1]], ref, "cont_batch full")
