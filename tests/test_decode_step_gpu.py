"""pkv_decode_step (append fused into the decode launch) through the C ABI:
bit-identical caches and outputs to pkv_kv_cache_append + pkv_paged_attn_decode,
and the oracle's append-then-decode within tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, oracle_decode, widen_out
from test_decode_gpu import SMALL

pytestmark = pytest.mark.gpu


def _two_call(pkv, w, d, kernel=0):
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    pkv.kv_cache_append(w.k_new.cuda(), w.v_new.cuda(), torch.from_numpy(w.slot_mapping).cuda(),
                        kc, vc)
    out = pkv.paged_attn_decode(d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                max_context_len=w.max_context_len, kernel=kernel)
    return out, kc, vc


def _fused(pkv, w, d, split_tokens=0, kernel=0):
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    out = pkv.decode_step(d["q"], w.k_new.cuda(), w.v_new.cuda(), kc, vc, d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len,
                          split_tokens=split_tokens, kernel=kernel)
    return out, kc, vc


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("name", W.ORDER)
def test_fused_step_matches_two_calls_and_oracle(pkv, name, seed):
    w = W.make(SMALL[name], seed=seed)
    d = device_inputs(w)
    o2, k2, v2 = _two_call(pkv, w, d)
    for split in (0, 16 if w.spec.block_size == 16 else 32):
        of, kf, vf = _fused(pkv, w, d, split)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert _same(kf, k2) and _same(vf, v2), "caches differ from append + decode"
        if split == 0:
            assert _same(of, o2), "output differs from append + decode"
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                           W.bits(w.k_cache), W.bits(w.v_cache))
    assert np.array_equal(W.bits(kf), ek) and np.array_equal(W.bits(vf), ev)
    assert_close(widen_out(of), oracle_decode(w, ek, ev), f"fused {name}/{seed}")


def test_fused_step_lengths_one_and_block_edges(pkv):
    lens = np.array([1, 16, 17, 32, 33, 1024, 1025], dtype=np.int32)
    for base in ("llama7b_mha", "llama3_8b_gqa", "long_ctx_gqa"):
        spec = W.scaled(W.WORKLOADS[base], len(lens), int(lens.max()))
        w = W.make(spec, seed=5, lens=lens)
        d = device_inputs(w)
        o2, k2, v2 = _two_call(pkv, w, d)
        of, kf, vf = _fused(pkv, w, d)
        torch.cuda.synchronize()
        assert _same(kf, k2) and _same(vf, v2) and _same(of, o2), base


def test_fused_step_full_continuous_batching(pkv):
    w = W.make("cont_batch", seed=0, device="cuda")
    d = device_inputs(w)
    o2, k2, v2 = _two_call(pkv, w, d)
    of, kf, vf = _fused(pkv, w, d)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert _same(kf, k2) and _same(vf, v2) and _same(of, o2)


@pytest.mark.parametrize("name", W.ORDER)
def test_fused_step_forced_partitions(pkv, name):
    """The append fused under short forced partitions (48 tokens, so the new
    token lands in the first, a middle or the last partition of a sequence):
    equal to append + decode bit for bit, caches included, and to the
    oracle."""
    w = W.make(SMALL[name], seed=7)
    d = device_inputs(w)
    kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
    pkv.kv_cache_append(w.k_new.cuda(), w.v_new.cuda(), torch.from_numpy(w.slot_mapping).cuda(),
                        kc2, vc2)
    o2 = pkv.paged_attn_decode(d["q"], kc2, vc2, d["block_tables"], d["context_lens"], w.scale,
                               max_context_len=w.max_context_len, split_tokens=48)
    of, kf, vf = _fused(pkv, w, d, split_tokens=48)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert _same(kf, kc2) and _same(vf, vc2) and _same(of, o2)
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                           W.bits(w.k_cache), W.bits(w.v_cache))
    assert np.array_equal(W.bits(kf), ek) and np.array_equal(W.bits(vf), ev)
    assert_close(widen_out(of), oracle_decode(w, ek, ev), f"forced-partition fused {name}")


@pytest.mark.parametrize("G", [4, 8, 32])
@pytest.mark.parametrize("bs", [16, 32])
def test_fused_step_tcgen05(pkv, G, bs):
    """The tcgen05 kernel's fused append: the new row reaches its cache slot
    and the staged K and V tiles; caches and output equal append + decode on
    the same kernel bit for bit, and the output matches the oracle.  Lengths
    put the new token at the start, middle and end of a 128-token group and
    of a block."""
    lens = np.array([1, 16, 17, 127, 128, 129, 300, 1024], dtype=np.int32)
    spec = W.WorkloadSpec("tcstep", len(lens), G * 2, 2, 128, bs, W.BF16, 0, 0, "uniform", (1, 1))
    spec = W.scaled(spec, len(lens), int(lens.max()))
    w = W.make(spec, seed=3 * G + bs, lens=lens)
    d = device_inputs(w)
    o2, k2, v2 = _two_call(pkv, w, d, kernel=3)
    of, kf, vf = _fused(pkv, w, d, kernel=3)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert _same(kf, k2) and _same(vf, v2), "caches differ from append + decode"
    assert _same(of, o2), "output differs from append + decode"
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                           W.bits(w.k_cache), W.bits(w.v_cache))
    assert np.array_equal(W.bits(kf), ek) and np.array_equal(W.bits(vf), ev)
    assert_close(widen_out(of), oracle_decode(w, ek, ev), f"tcgen05 fused G={G} bs={bs}")


@pytest.mark.parametrize("G", [12, 32])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32), (128, 32)])
@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_fused_step_wide_groups(pkv, G, D, bs, dtype):
    """Wide query groups on mma.sync (warp pairs where the stages are 8 KB or
    less: the first warp of a pair writes the new row into the staged tile,
    the second waits for it): caches and output equal append + decode bit for
    bit, with automatic and short forced partitions, and match the oracle.
    Lengths put the new token at the start, middle and end of a block."""
    lens = np.array([1, bs, bs + 1, 2 * bs - 1, 300, 777, 1500], dtype=np.int32)
    spec = W.WorkloadSpec("widestep", len(lens), G * 2, 2, D, bs, dtype, 0, 0, "uniform", (1, 1))
    spec = W.scaled(spec, len(lens), int(lens.max()))
    w = W.make(spec, seed=5 * G + D + bs, lens=lens)
    d = device_inputs(w)
    ek, ev = oracle.append(W.bits(w.k_new), W.bits(w.v_new), w.slot_mapping,
                           W.bits(w.k_cache), W.bits(w.v_cache))
    ref = oracle_decode(w, ek, ev)
    for split in (0, 3 * bs):
        kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
        pkv.kv_cache_append(w.k_new.cuda(), w.v_new.cuda(),
                            torch.from_numpy(w.slot_mapping).cuda(), kc2, vc2)
        o2 = pkv.paged_attn_decode(d["q"], kc2, vc2, d["block_tables"], d["context_lens"],
                                   w.scale, max_context_len=w.max_context_len,
                                   split_tokens=split)
        of, kf, vf = _fused(pkv, w, d, split_tokens=split)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert _same(kf, kc2) and _same(vf, vc2) and _same(of, o2), f"G={G} D={D} split={split}"
        assert np.array_equal(W.bits(kf), ek) and np.array_equal(W.bits(vf), ev)
        assert_close(widen_out(of), ref, f"wide fused G={G} D={D} bs={bs} split={split}")
