"""Randomised parity sweep through the C ABI: seeded random shapes (head_dim,
block size, group size, kv heads, batch, dtype), ragged lengths (1 token,
block edges, several partitions), partition sizes (the library's choice,
one block, odd forced sizes), kernels (the library's choice and tcgen05 at
head_dim 128) and both entry points (plain decode, fused append + decode),
each against the oracle: caches bit-exact after the fused step, outputs
within the parity tolerance, the device error word clear."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, oracle_decode, widen_out

pytestmark = pytest.mark.gpu

CASES = 120


def _case(rng: np.random.Generator, i: int):
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32]))
    G = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    if G * Hkv > 128:
        Hkv = max(1, 128 // G)
    B = int(rng.integers(1, 9))
    dtype = int(rng.choice([W.F16, W.BF16]))
    kernel = int(rng.choice([0, 0, 3])) if D == 128 else 0
    maxlen = int(rng.choice([1, 15, 16, 17, 100, 700, 1500, 2600]))
    lens = rng.integers(1, maxlen + 1, size=B).astype(np.int32)
    lens[0] = maxlen
    split = int(rng.choice([0, 0, bs, 3 * bs, int(rng.integers(1, 3000))]))
    fused = bool(rng.integers(0, 2))
    spec = W.WorkloadSpec("rand", B, G * Hkv, Hkv, D, bs, dtype, 0, 0, "uniform", (1, 1))
    spec = W.scaled(spec, B, int(lens.max()))
    w = W.make(spec, seed=i, lens=lens)
    desc = (f"case {i}: D={D} bs={bs} G={G} Hkv={Hkv} B={B} dtype={dtype} kernel={kernel} "
            f"lens={lens.tolist()} split={split} fused={fused}")
    return w, kernel, split, fused, desc


@pytest.mark.parametrize("block", range(4))
def test_random_shapes_match_the_oracle(pkv, block):
    rng = np.random.default_rng([2027, block])
    for i in range(CASES // 4):
        w, kernel, split, fused, desc = _case(rng, block * 1000 + i)
        d = device_inputs(w)
        if fused:
            kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
            out = pkv.decode_step(d["q"], w.k_new.cuda(), w.v_new.cuda(), kc, vc,
                                  d["block_tables"], d["context_lens"], w.scale,
                                  max_context_len=w.max_context_len, split_tokens=split,
                                  kernel=kernel)
            torch.cuda.synchronize()
            ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                                   W.bits(w.k_cache), W.bits(w.v_cache))
            assert np.array_equal(W.bits(kc), ek) and np.array_equal(W.bits(vc), ev), desc
            ref = oracle_decode(w, ek, ev)
        else:
            out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                        d["context_lens"], w.scale,
                                        max_context_len=w.max_context_len, split_tokens=split,
                                        kernel=kernel)
            torch.cuda.synchronize()
            ref = oracle_decode(w)
        assert pkv.get_device_error() == 0, desc
        assert_close(widen_out(out), ref, desc)
