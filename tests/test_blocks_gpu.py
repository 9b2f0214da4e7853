"""pkv_copy_blocks and the block manager driving real decode steps (GPU).

Block copies are bit-exact against the oracle between device pools and
between a device pool and a pinned host pool.  The end-to-end test runs a
small continuous-batching session: prefill by slot scatter, forked sequences
sharing prefix blocks, copy-on-write, swap-out to and swap-in from pinned CPU
memory, sequences leaving, and fused decode steps, mirrored on the host with
the oracle after every step."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, widen_out

pytestmark = pytest.mark.gpu


def _pool(nb, hkv, bs, d, dtype, gen, device="cuda", pinned=False):
    t = torch.randn((nb, hkv, bs, d), generator=gen).to(dtype)
    return t.pin_memory() if pinned else t.to(device)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_copy_blocks_device_and_pinned_host(pkv, dtype):
    g = torch.Generator().manual_seed(1)
    hkv, bs, d = 8, 16, 128
    gk, gv = _pool(40, hkv, bs, d, dtype, g), _pool(40, hkv, bs, d, dtype, g)
    ck, cv = _pool(25, hkv, bs, d, dtype, g, pinned=True), _pool(25, hkv, bs, d, dtype, g, pinned=True)
    # device -> device (copy-on-write), pairs in device memory
    pairs = torch.tensor([[3, 10], [39, 0], [7, 21]], dtype=torch.int32)
    k0, v0 = W.bits(gk), W.bits(gv)
    pkv.copy_blocks(gk, gv, gk, gv, pairs.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(gk), oracle.copy_blocks(k0, k0, pairs.numpy()))
    assert np.array_equal(W.bits(gv), oracle.copy_blocks(v0, v0, pairs.numpy()))
    # device -> pinned host (swap out), pairs in pinned host memory
    out_pairs = torch.tensor([[0, 24], [5, 0], [39, 13]], dtype=torch.int32).pin_memory()
    hk0, hv0 = W.bits(ck), W.bits(cv)
    pkv.copy_blocks(gk, gv, ck, cv, out_pairs)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(ck), oracle.copy_blocks(W.bits(gk), hk0, out_pairs.numpy()))
    assert np.array_equal(W.bits(cv), oracle.copy_blocks(W.bits(gv), hv0, out_pairs.numpy()))
    # pinned host -> device (swap in)
    in_pairs = torch.tensor([[24, 1], [13, 2]], dtype=torch.int32).cuda()
    k1 = W.bits(gk)
    pkv.copy_blocks(ck, cv, gk, gv, in_pairs)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(gk), oracle.copy_blocks(W.bits(ck), k1, in_pairs.cpu().numpy()))
    assert pkv.get_device_error() == 0


def test_copy_blocks_bad_pair_sets_device_error(pkv):
    g = torch.Generator().manual_seed(2)
    gk, gv = _pool(8, 2, 16, 64, torch.float16, g), _pool(8, 2, 16, 64, torch.float16, g)
    before = W.bits(gk)
    pairs = torch.tensor([[1, 2], [9, 3], [4, -1], [5, 6]], dtype=torch.int32).cuda()
    pkv.copy_blocks(gk, gv, gk, gv, pairs)
    assert pkv.get_device_error() == 1
    exp = oracle.copy_blocks(before, before, np.array([[1, 2], [5, 6]], dtype=np.int32))
    assert np.array_equal(W.bits(gk), exp)          # the good pairs were copied


def test_continuous_batching_session_with_allocator(pkv):
    rng = np.random.default_rng(7)
    g = torch.Generator().manual_seed(7)
    hkv, G, bs, d, dtype = 4, 2, 16, 128, torch.float16
    NG, NC, MB = 160, 64, 40
    scale = float(np.float32(1 / np.sqrt(d)))
    kc = torch.full((NG, hkv, bs, d), float("nan"), dtype=dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    hk = torch.zeros((NC, hkv, bs, d), dtype=dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    mk, mv = W.bits(kc), W.bits(vc)               # host mirrors
    mhk, mhv = W.bits(hk), W.bits(hv)
    m = pkv.BlockManager(NG, NC, bs)

    def rows(n):
        return torch.randn((n, hkv, d), generator=g).to(dtype)

    def scatter(k, v, slots):
        nonlocal mk, mv
        pkv.kv_cache_append(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), kc, vc)
        mk, mv = oracle.append(W.bits(k), W.bits(v), slots, mk, mv)

    def copy(pairs, direction):
        nonlocal mk, mv, mhk, mhv
        if len(pairs) == 0:
            return
        p = torch.from_numpy(np.ascontiguousarray(pairs, dtype=np.int32)).cuda()
        if direction == "gg":
            pkv.copy_blocks(kc, vc, kc, vc, p)
            mk, mv = oracle.copy_blocks(mk, mk, pairs), oracle.copy_blocks(mv, mv, pairs)
        elif direction == "gc":
            pkv.copy_blocks(kc, vc, hk, hv, p)
            mhk, mhv = oracle.copy_blocks(mk, mhk, pairs), oracle.copy_blocks(mv, mhv, pairs)
        else:
            pkv.copy_blocks(hk, hv, kc, vc, p)
            mk, mv = oracle.copy_blocks(mhk, mk, pairs), oracle.copy_blocks(mhv, mv, pairs)

    # prefill: three prompts written through their slots
    live = []
    for sid, n in enumerate(rng.integers(20, 250, size=3)):
        m.add_sequence(sid, int(n))
        t, _ = m.block_tables([sid], MB)
        pos = np.arange(int(n))
        scatter(rows(int(n)), rows(int(n)), (t[0, pos // bs] * bs + pos % bs).astype(np.int32))
        live.append(sid)
    # two forks of sequence 0 share its blocks (prefix reuse)
    for child in (10, 11):
        m.fork(0, child)
        live.append(child)
    swapped = None
    for step in range(14):
        if step == 4:                              # sequence 1 leaves the GPU for a while
            copy(m.swap_out(1, 2), "gc")
            live.remove(1)
            swapped = 1
        if step == 9:                              # ... and comes back
            copy(m.swap_in(swapped), "cg")
            live.append(swapped)
        if step == 7:                              # sequence 2 finishes
            m.free_sequence(2)
            live.remove(2)
        cow, slots = [], []
        for sid in live:
            slot, cs, cd = m.append_token(sid)
            slots.append(slot)
            if cs >= 0:
                cow.append((cs, cd))
        copy(np.array(cow, dtype=np.int32).reshape(-1, 2), "gg")
        t, lens = m.block_tables(live, MB)
        derived = t[np.arange(len(live)), (lens - 1) // bs] * bs + (lens - 1) % bs
        assert derived.tolist() == slots           # the fused step's slot rule agrees
        q = torch.randn((len(live), hkv * G, d), generator=g).to(dtype)
        kn, vn = rows(len(live)), rows(len(live))
        out = pkv.decode_step(q.cuda(), kn.cuda(), vn.cuda(), kc, vc,
                              torch.from_numpy(t).cuda(), torch.from_numpy(lens).cuda(), scale,
                              max_context_len=MB * bs)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        mk, mv = oracle.append(W.bits(kn), W.bits(vn), np.array(slots, dtype=np.int32), mk, mv)
        ref = oracle.decode(W.bits(q), mk, mv, t, lens, scale, W.F16)
        assert_close(widen_out(out), ref, f"step {step}")
    # the device pools equal their host mirrors, block by block
    assert np.array_equal(W.bits(kc), mk) and np.array_equal(W.bits(vc), mv)
    assert np.array_equal(W.bits(hk), mhk)
    m.close()
