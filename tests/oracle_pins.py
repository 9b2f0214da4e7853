"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (a closed form, a hand-worked value, a library routine on unpaged data,
an exhaustive format table, an invariance).  Every check takes the ctypes
handle of an oracle build, so the same checks also run against deliberately
broken copies of the oracle (tests/test_oracle_mutants.py) to show that a
plausible mistake fails at least one of them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F16, BF16 = oracle.F16, oracle.BF16


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.to(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _from_bits(b: np.ndarray, dtype: int) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16))
    t = t.view(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.to(torch.float64).numpy()


def page(kc_contig: np.ndarray, bs: int, table: np.ndarray, NB: int, fill=0x7FC0):
    """Scatter contiguous per-sequence K or V [B][Hkv][L][D] (ragged list) into a
    paged pool [NB, Hkv, bs, D] following ``table`` (test-side layout helper).
    Unreferenced rows get 0x7FC0, a NaN in both binary16 and bfloat16."""
    B = len(kc_contig)
    Hkv, _, D = kc_contig[0].shape
    pool = np.full((NB, Hkv, bs, D), fill, dtype=np.uint16)
    for i in range(B):
        L = kc_contig[i].shape[1]
        for t in range(L):
            pool[table[i, t // bs], :, t % bs, :] = kc_contig[i][:, t, :]
    return pool


def _case(rng, B, Hq, Hkv, D, bs, lens, dtype, NB=None, perm=True, k_scale=1.0):
    lens = np.asarray(lens, dtype=np.int32)
    MB = int(-(-lens.max() // bs))
    need = int(sum(-(-int(L) // bs) for L in lens))
    NB = NB or need + 3
    ids = rng.permutation(NB) if perm else np.arange(NB)
    table = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for i, L in enumerate(lens):
        n = -(-int(L) // bs)
        table[i, :n] = ids[k:k + n]
        k += n
    q = _to_bits(rng.standard_normal((B, Hq, D)), dtype)
    kc = [_to_bits(k_scale * rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    vc = [_to_bits(rng.standard_normal((Hkv, int(L), D)), dtype) for L in lens]
    return dict(q=q, kc=kc, vc=vc, table=table, lens=lens, NB=NB, bs=bs)


def _sdpa(q_bits, k_bits, v_bits, scale, dtype):
    """torch's attention routine on unpaged fp64 data (library reference)."""
    q = torch.from_numpy(_from_bits(q_bits, dtype))[None, None, None, :]
    k = torch.from_numpy(_from_bits(k_bits, dtype))[None, None]
    v = torch.from_numpy(_from_bits(v_bits, dtype))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)[0, 0, 0].numpy()


# ---------------------------------------------------------------- formats
def check_half_decode_exhaustive(lib):
    """All 65536 binary16 patterns widen exactly as numpy's float16 does."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(pats, F16, lib)
    ref = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, got[0x8000]) == -1.0


def check_bf16_decode_exhaustive(lib):
    """All 65536 bfloat16 patterns widen exactly as torch's bfloat16 does."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(pats, BF16, lib)
    ref = _from_bits(pats, BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- closed forms
def check_hand_worked(lib):
    g = _read_golden("hand_worked_softmax.txt")
    D = int(g["head_dim"][0])
    for dtype in (F16, BF16):
        for bs, perm in ((16, False), (2, True), (1, True)):
            rng = np.random.default_rng(7)
            q = np.zeros((1, 1, D)); q[0, 0, 0] = g["q0"][0]
            kcont = np.zeros((1, 3, D)); kcont[0, :, 0] = g["k0"]
            vcont = np.zeros((1, 3, D)); vcont[0, :, 0] = g["v0"]
            c = _case(rng, 1, 1, 1, D, bs, [3], dtype, perm=perm)
            kc = page([_to_bits(kcont, dtype)], bs, c["table"], c["NB"])
            vc = page([_to_bits(vcont, dtype)], bs, c["table"], c["NB"])
            out = oracle.decode(_to_bits(q, dtype), kc, vc, c["table"], c["lens"],
                                g["scale"][0], dtype, lib)
            assert abs(out[0, 0, 0] - g["out0"][0]) <= 1e-15, out[0, 0, 0]
            assert np.all(out[0, 0, 1:] == 0.0)


def check_two_token_logistic(lib):
    g = _read_golden("two_token_logistic.txt")
    D = int(g["head_dim"][0])
    q = np.zeros((1, 1, D)); q[0, 0, 3] = 1.5
    kcont = np.zeros((1, 2, D)); kcont[0, 1, 3] = 2.0
    vcont = np.zeros((1, 2, D)); vcont[0, 1, 5] = 1.0
    for dtype in (F16, BF16):
        c = _case(np.random.default_rng(1), 1, 1, 1, D, 16, [2], dtype)
        kc = page([_to_bits(kcont, dtype)], 16, c["table"], c["NB"])
        vc = page([_to_bits(vcont, dtype)], 16, c["table"], c["NB"])
        out = oracle.decode(_to_bits(q, dtype), kc, vc, c["table"], c["lens"],
                            g["scale"][0], dtype, lib)
        assert abs(out[0, 0, 5] - g["out5"][0]) <= 1e-15
        expect = np.zeros(D); expect[5] = g["out5"][0]
        assert np.allclose(out[0, 0], expect, atol=1e-15, rtol=0)


def check_single_token_returns_v(lib):
    """context_len 1: the only softmax weight is 1, so out = v_0 exactly."""
    for dtype in (F16, BF16):
        rng = np.random.default_rng(3)
        c = _case(rng, 3, 4, 2, 64, 16, [1, 1, 1], dtype)
        kc = page(c["kc"], 16, c["table"], c["NB"])
        vc = page(c["vc"], 16, c["table"], c["NB"])
        out = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.3, dtype, lib)
        for i in range(3):
            for h in range(4):
                v0 = _from_bits(c["vc"][i][h // 2, 0], dtype)
                assert np.array_equal(out[i, h], v0)


def check_constant_k_gives_mean_v(lib):
    """All k_t equal: uniform softmax, out = mean_t v_t."""
    for dtype in (F16, BF16):
        rng = np.random.default_rng(4)
        lens = [5, 16, 33]
        c = _case(rng, 3, 2, 1, 64, 16, lens, dtype)
        krow = _to_bits(rng.standard_normal(64), dtype)
        kcs = [np.broadcast_to(krow, (1, L, 64)).copy() for L in lens]
        kc = page(kcs, 16, c["table"], c["NB"])
        vc = page(c["vc"], 16, c["table"], c["NB"])
        out = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.7, dtype, lib)
        for i in range(3):
            mean = _from_bits(c["vc"][i][0], dtype).mean(axis=0)
            for h in range(2):
                assert np.allclose(out[i, h], mean, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- library routine
def check_matches_library_attention(lib):
    """Random paged batches equal torch's scaled_dot_product_attention run on
    the same data before it was paged (GQA heads mapped h -> h // G)."""
    for dtype, Hq, Hkv, bs in ((F16, 4, 4, 16), (BF16, 8, 2, 32), (F16, 6, 2, 16)):
        rng = np.random.default_rng(10 + Hq)
        lens = [1, 15, 16, 17, 70]
        c = _case(rng, 5, Hq, Hkv, 64, bs, lens, dtype)
        kc = page(c["kc"], bs, c["table"], c["NB"])
        vc = page(c["vc"], bs, c["table"], c["NB"])
        scale = 0.125
        out = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], scale, dtype, lib)
        G = Hq // Hkv
        for i in range(5):
            for h in range(Hq):
                ref = _sdpa(c["q"][i, h], c["kc"][i][h // G], c["vc"][i][h // G], scale, dtype)
                assert np.allclose(out[i, h], ref, rtol=1e-12, atol=1e-13), (i, h)


def check_identity_table_matches_library(lib):
    """Identity block table (logical block j of seq i -> i*MB + j) vs the
    library routine on the contiguous data."""
    dtype, bs = BF16, 16
    rng = np.random.default_rng(21)
    lens = [40, 64]
    c = _case(rng, 2, 2, 2, 64, bs, lens, dtype, perm=False)
    MB = c["table"].shape[1]
    table = np.arange(2 * MB, dtype=np.int32).reshape(2, MB)
    kc = page(c["kc"], bs, table, 2 * MB)
    vc = page(c["vc"], bs, table, 2 * MB)
    out = oracle.decode(c["q"], kc, vc, table, c["lens"], 0.2, dtype, lib)
    for i in range(2):
        for h in range(2):
            ref = _sdpa(c["q"][i, h], c["kc"][i][h], c["vc"][i][h], 0.2, dtype)
            assert np.allclose(out[i, h], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- invariances
def check_permutation_invariance(lib):
    """Relabelling physical blocks (data moved with the ids) leaves the output
    bit-identical; the summation order does not change."""
    dtype, bs = F16, 16
    rng = np.random.default_rng(5)
    c = _case(rng, 3, 4, 4, 64, bs, [20, 48, 33], dtype)
    kc = page(c["kc"], bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    out1 = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.1, dtype, lib)
    sigma = rng.permutation(c["NB"])           # new id of old block b is sigma[b]
    kc2 = np.empty_like(kc); kc2[sigma] = kc
    vc2 = np.empty_like(vc); vc2[sigma] = vc
    t2 = np.where(c["table"] >= 0, sigma[np.maximum(c["table"], 0)], -1).astype(np.int32)
    out2 = oracle.decode(c["q"], kc2, vc2, t2, c["lens"], 0.1, dtype, lib)
    assert np.array_equal(out1, out2)


def check_gqa_equals_repeated_mha(lib):
    """GQA with group G equals MHA whose kv heads are each repeated G times."""
    dtype, bs, G, Hkv = BF16, 16, 4, 2
    rng = np.random.default_rng(6)
    c = _case(rng, 2, G * Hkv, Hkv, 64, bs, [19, 40], dtype)
    kc = page(c["kc"], bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    gqa = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.15, dtype, lib)
    kr, vr = np.repeat(kc, G, axis=1), np.repeat(vc, G, axis=1)
    mha = oracle.decode(c["q"], kr, vr, c["table"], c["lens"], 0.15, dtype, lib)
    assert np.array_equal(gqa, mha)


def check_softmax_shift_invariance(lib):
    """Adding the same constant to every logit leaves the output unchanged:
    every k_t has the same last component c, so moving q's last component
    shifts all logits of the row by the same amount."""
    dtype, bs = F16, 16
    rng = np.random.default_rng(8)
    c = _case(rng, 1, 1, 1, 64, bs, [37], dtype)
    kcs = [c["kc"][0].copy()]
    kcs[0][..., 63] = _to_bits(np.full((1, 37), 0.5), dtype)
    kc = page(kcs, bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    q1 = c["q"].copy()
    q2 = c["q"].copy(); q2[..., 63] = _to_bits(np.array([3.0]), dtype)
    q1[..., 63] = _to_bits(np.array([-2.0]), dtype)
    o1 = oracle.decode(q1, kc, vc, c["table"], c["lens"], 0.5, dtype, lib)
    o2 = oracle.decode(q2, kc, vc, c["table"], c["lens"], 0.5, dtype, lib)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12)
    # ... and the shift is not a no-op for a k that varies in that component
    kcs[0][..., 63] = _to_bits(rng.standard_normal((1, 37)), dtype)
    kc3 = page(kcs, bs, c["table"], c["NB"])
    o3 = oracle.decode(q1, kc3, vc, c["table"], c["lens"], 0.5, dtype, lib)
    o4 = oracle.decode(q2, kc3, vc, c["table"], c["lens"], 0.5, dtype, lib)
    assert not np.allclose(o3, o4, rtol=0, atol=1e-6)


def check_rows_match_batch(lib):
    """The sampled-row entry point returns the same rows as the batch one."""
    dtype, bs = BF16, 32
    rng = np.random.default_rng(9)
    c = _case(rng, 3, 8, 2, 64, bs, [31, 32, 90], dtype)
    kc = page(c["kc"], bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    full = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.3, dtype, lib)
    rows = [(0, 0), (2, 7), (1, 3), (2, 4)]
    part = oracle.decode_rows(rows, c["q"], kc, vc, c["table"], c["lens"], 0.3, dtype, lib)
    for r, (i, h) in enumerate(rows):
        assert np.array_equal(part[r], full[i, h])


def check_scale_enters_logits(lib):
    """scale multiplies the logits: scale 0 gives the plain mean of V, and
    doubling the scale equals doubling q (exact in binary floating point)."""
    dtype, bs = F16, 16
    rng = np.random.default_rng(11)
    c = _case(rng, 1, 1, 1, 64, bs, [29], dtype)
    kc = page(c["kc"], bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    o0 = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.0, dtype, lib)
    assert np.allclose(o0[0, 0], _from_bits(c["vc"][0][0], dtype).mean(axis=0), atol=1e-12, rtol=0)
    q = _from_bits(c["q"], dtype)
    q2 = _to_bits(2 * q, dtype)
    assert np.array_equal(_from_bits(q2, dtype), 2 * q)
    oa = oracle.decode(c["q"], kc, vc, c["table"], c["lens"], 0.25, dtype, lib)
    ob = oracle.decode(q2, kc, vc, c["table"], c["lens"], 0.125, dtype, lib)
    assert np.allclose(oa, ob, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- append
def check_append_matches_index_assignment(lib):
    """The append scatter equals numpy fancy-index assignment of the new rows
    into the pool; negative slots write nothing; other slots stay unchanged."""
    rng = np.random.default_rng(12)
    NB, Hkv, bs, D, T = 9, 3, 16, 64, 11
    kc = rng.integers(0, 65536, size=(NB, Hkv, bs, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(NB, Hkv, bs, D), dtype=np.uint16)
    k = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int32)
    slots[[2, 7]] = -1
    kc2, vc2 = oracle.append(k, v, slots, kc, vc, lib)
    ek, ev = kc.copy(), vc.copy()
    ok = slots >= 0
    ek[slots[ok] // bs, :, slots[ok] % bs, :] = k[ok]
    ev[slots[ok] // bs, :, slots[ok] % bs, :] = v[ok]
    assert np.array_equal(kc2, ek) and np.array_equal(vc2, ev)
    # input arrays untouched (the wrapper works on copies)
    assert not np.array_equal(kc2, kc)


def check_append_then_decode_sees_token(lib):
    """After appending a token with a huge logit, decode returns its v row."""
    dtype, bs = F16, 16
    rng = np.random.default_rng(13)
    c = _case(rng, 1, 1, 1, 64, bs, [24], dtype)
    kc = page(c["kc"], bs, c["table"], c["NB"])
    vc = page(c["vc"], bs, c["table"], c["NB"])
    q = np.zeros((1, 1, 64)); q[0, 0, 0] = 1.0
    knew = np.zeros((1, 1, 64)); knew[0, 0, 0] = 1000.0
    vnew = rng.standard_normal((1, 1, 64))
    pos = 23
    slot = np.array([c["table"][0, pos // bs] * bs + pos % bs], dtype=np.int32)
    kc2, vc2 = oracle.append(_to_bits(knew, dtype), _to_bits(vnew, dtype), slot, kc, vc, lib)
    out = oracle.decode(_to_bits(q, dtype), kc2, vc2, c["table"], c["lens"], 1.0, dtype, lib)
    assert np.allclose(out[0, 0], _from_bits(_to_bits(vnew, dtype), dtype)[0, 0], atol=1e-12, rtol=0)


def check_copy_blocks_matches_index_assignment(lib):
    """Block copy equals numpy fancy-index assignment between pools of
    different sizes; blocks not named as destinations stay unchanged."""
    rng = np.random.default_rng(14)
    src = rng.integers(0, 65536, size=(7, 2, 16, 64), dtype=np.uint16)
    dst = rng.integers(0, 65536, size=(11, 2, 16, 64), dtype=np.uint16)
    pairs = np.array([[3, 0], [6, 10], [0, 4], [3, 7]], dtype=np.int32)
    got = oracle.copy_blocks(src, dst, pairs, lib)
    exp = dst.copy()
    exp[pairs[:, 1]] = src[pairs[:, 0]]
    assert np.array_equal(got, exp)


ALL_CHECKS = [
    check_half_decode_exhaustive,
    check_bf16_decode_exhaustive,
    check_hand_worked,
    check_two_token_logistic,
    check_single_token_returns_v,
    check_constant_k_gives_mean_v,
    check_matches_library_attention,
    check_identity_table_matches_library,
    check_permutation_invariance,
    check_gqa_equals_repeated_mha,
    check_softmax_shift_invariance,
    check_rows_match_batch,
    check_scale_enters_logits,
    check_append_matches_index_assignment,
    check_append_then_decode_sees_token,
    check_copy_blocks_matches_index_assignment,
]
