"""The seeded input recipe (CPU only): lengths, block tables, prefix sharing,
slot mapping and canary fill follow the stated recipe."""
import numpy as np
import pytest
import torch

from paged_kv_cache_268_gb300 import workloads as W


@pytest.mark.parametrize("name", W.ORDER)
def test_lengths_and_tables(name):
    spec = W.WORKLOADS[name]
    rng = np.random.default_rng([0, W.ORDER.index(name)])
    lens = W.context_lengths(spec, rng)
    tables, used = W.block_tables(spec, lens, rng)
    bs = spec.block_size
    assert lens.shape == (spec.num_seqs,)
    nblk = -(-lens // bs)
    assert nblk.max() <= spec.max_blocks_per_seq
    owners = {}
    for i in range(spec.num_seqs):
        row = tables[i]
        assert np.all(row[:nblk[i]] >= 0) and np.all(row[:nblk[i]] < spec.num_blocks)
        assert np.all(row[nblk[i]:] == -1)
        for j, p in enumerate(row[:nblk[i]]):
            owners.setdefault(int(p), []).append((i, j))
    assert used.sum() == len(owners)
    for p, users in owners.items():
        if len(users) > 1:
            # only the continuous-batching workload shares, and only prefix blocks
            assert spec.share_prefix
            js = {j for _, j in users}
            groups = {i // 8 for i, _ in users}
            assert len(js) == 1 and len(groups) == 1 and next(iter(js)) < 32
    if name == "tiny_mha":
        assert list(lens) == [1, 17, 64, 200] and used.sum() == 20
    if name == "long_ctx_gqa":
        assert np.all(lens == 32768) and used.sum() == 4096
    if name == "llama3_8b_gqa":
        assert lens.min() >= 16 and lens.max() <= 8192
    if spec.share_prefix:
        nshared = np.minimum(32, (lens - 1) // bs)
        for i in range(spec.num_seqs):
            lead = (i // 8) * 8
            ns = min(nshared[i], nshared[lead])
            assert np.array_equal(tables[i, :ns], tables[lead, :ns])


@pytest.mark.parametrize("name", W.ORDER)
def test_append_slots_are_private_and_last(name):
    spec = W.WORKLOADS[name]
    rng = np.random.default_rng([1, W.ORDER.index(name)])
    lens = W.context_lengths(spec, rng)
    tables, _ = W.block_tables(spec, lens, rng)
    slots = W.append_slots(spec, lens, tables)
    assert len(set(slots.tolist())) == spec.num_seqs        # unique slots
    blk, off = slots // spec.block_size, slots % spec.block_size
    assert np.array_equal(off, (lens - 1) % spec.block_size)
    # the block receiving the new token is referenced by exactly one sequence
    for i in range(spec.num_seqs):
        assert (tables == blk[i]).sum() == 1


def test_make_small_is_seeded_and_poisoned():
    a = W.make("tiny_mha", seed=0)
    b = W.make("tiny_mha", seed=0)
    c = W.make("tiny_mha", seed=1)
    assert np.array_equal(W.bits(a.k_cache), W.bits(b.k_cache))
    assert np.array_equal(W.bits(a.q), W.bits(b.q))
    assert not np.array_equal(W.bits(a.k_cache), W.bits(c.k_cache))
    kb = W.bits(a.k_cache)
    assert np.all(kb[~a.used_blocks] == W.NAN_BITS[W.F16])
    assert not np.any(kb[a.used_blocks] == W.NAN_BITS[W.F16])
    assert a.kv_bytes() == 577536
    assert a.q.dtype == torch.float16 and a.q.shape == (4, 8, 64)


def test_scaled_spec_and_k_spread():
    spec = W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 300, lens="fixed")
    w = W.make(spec, seed=3)
    assert list(w.context_lens) == [300, 300]
    k = w.k_cache.float()[torch.from_numpy(w.used_blocks)]
    row_rms = k.pow(2).mean(-1).sqrt()
    assert row_rms.min() < 0.75 and row_rms.max() > 1.5   # U(0.5, 2) row spread
    assert w.k_cache.dtype == torch.bfloat16
