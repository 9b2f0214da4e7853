"""Host-side split-KV planning, CPU only: pkv_decode_plan_for plans a decode
call for a given SM count without touching a GPU.

The partition schedule gives every (sequence, kv head, partition of P tokens)
one CTA (the tiling of the third page, "FlashAttention deep integration",
over the paged layout of its "PagedAttention" section).  This file restates
the planner's documented rule and launch geometry in Python and checks the
library against it on a sweep of shapes and SM counts, plus the benchmark
workloads' plans as worked examples."""
from __future__ import annotations

import ctypes
import itertools

import numpy as np
import pytest

from paged_kv_cache_268_gb300 import _binding as B
from paged_kv_cache_268_gb300 import build
from paged_kv_cache_268_gb300 import workloads as W

GB300_SMS = 152
MAX_BLOCKS_PER_CTA = 256
ERR_NULL, ERR_INVALID, ERR_UNSUPPORTED = -1, -2, -3     # PKV_ERR_* of include/pkv.h


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load_library()


# ------------------------------------------------------------ restated geometry
def stage_bytes(D, bs):
    return 2 * bs * D * 2                      # a K tile and a V tile of 16-bit elements


def warps(D, bs):
    sb = stage_bytes(D, bs)
    return 4 if sb <= 8192 else (2 if sb <= 16384 else 1)


def heads_per_warp(variant, G):
    return G if variant == 0 else 8 * (1 if G <= 8 else (2 if G <= 16 else 4))


def stages(D, bs, nh):
    return 3 if warps(D, bs) == 4 and nh * D >= 2048 else 2


def smem(D, bs, nh):
    nw, ns = warps(D, bs), stages(D, bs, nh)
    ring = nw * ns * stage_bytes(D, bs)
    merge = nw * nh * (D + 2) * 4
    extra = ((merge - ring + 15) & ~15) if merge > ring else 0
    return ring + nw * ns * 8 + MAX_BLOCKS_PER_CTA * 4 + 1024 + extra


def ctas_per_sm(nbytes):
    return min(233472 // (nbytes + 1024), 16)  # 228 KB per SM, 1 KB reserved per CTA


def expected_plan(B_, Hq, Hkv, D, bs, maxL, split, sms):
    """(variant, P, S, grid, workspace bytes) of the partition schedule for
    the CUDA-core and mma.sync kernels."""
    G = Hq // Hkv
    variant = 0 if G <= 2 else 1
    nh = heads_per_warp(variant, G)
    nw = warps(D, bs)
    gran = bs * nw
    cap = MAX_BLOCKS_PER_CTA * bs
    units = B_ * Hkv
    if split > 0:
        P = -(-split // bs) * bs
    else:
        wide = variant == 1 and G > 8
        P = 2048 if wide else 1024
        cps = ctas_per_sm(smem(D, bs, nh))
        slots = sms * cps
        if units > 0 and units * -(-maxL // P) < (2 if wide else 4) * slots:
            # one wave; the two-warp CTAs (16 KB stages) fill it at two per SM
            wave = 2 * sms if nw == 2 and cps > 2 else slots
            S = max(wave // units, 1)
            P = -(-maxL // S)
        P = -(-P // gran) * gran
        pmin = -(-maxL // 1024)                 # at most 1024 partitions per sequence
        if P < pmin:
            P = -(-pmin // gran) * gran
    P = min(P, cap)
    if P > maxL:
        P = -(-maxL // bs) * bs
    P = max(P, bs)
    S = -(-maxL // P)
    ws = B_ * Hq * S * (D * 4 + 8) if S > 1 else 0
    return variant, P, S, units * S, ws


def plan_for(lib, sms, **kw):
    base = dict(num_seqs=1, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16,
                num_blocks=1024, max_blocks_per_seq=1, max_context_len=1, dtype=B.PKV_F16)
    base.update(kw)
    if "max_blocks_per_seq" not in kw:
        base["max_blocks_per_seq"] = -(-base["max_context_len"] // base["block_size"])
    return B.decode_plan(B.make_shape(**base), num_sms=sms)


# ------------------------------------------------------------ worked examples
def test_benchmark_workload_plans(lib):
    """The plans the benchmark workloads get on a 152-SM GB300."""
    want = {  # workload: (variant, P, S, grid)
        "llama7b_mha": (0, 1024, 4, 64 * 32 * 4),
        "llama3_8b_gqa": (1, 1024, 8, 128 * 8 * 8),
        "long_ctx_gqa": (1, 3648, 9, 4 * 8 * 9),         # one wave at two CTAs per SM
        "cont_batch": (1, 1024, 2, 256 * 8 * 2),
        "tiny_mha": (0, 64, 4, 4 * 8 * 4),               # one wave, rounded to the 64-token grain
        "wide_gqa16": (1, 2048, 2, 64 * 8 * 2),
        "wide_gqa32": (1, 2048, 2, 64 * 8 * 2),
    }
    maxlen = {"llama7b_mha": 4096, "llama3_8b_gqa": 8192, "long_ctx_gqa": 32768,
              "cont_batch": 2048, "tiny_mha": 200, "wide_gqa16": 4096, "wide_gqa32": 4096}
    for name, (variant, P, S, grid) in want.items():
        spec = W.WORKLOADS[name]
        p = plan_for(lib, GB300_SMS, num_seqs=spec.num_seqs, num_q_heads=spec.num_q_heads,
                     num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                     block_size=spec.block_size, num_blocks=spec.num_blocks,
                     max_blocks_per_seq=spec.max_blocks_per_seq, max_context_len=maxlen[name],
                     dtype=spec.dtype)
        assert (p.schedule, p.variant, p.split_tokens, p.num_splits, p.grid_ctas) == \
            (0, variant, P, S, grid), name
        rows = spec.num_seqs * spec.num_q_heads * S
        assert p.workspace_bytes == rows * (spec.head_dim * 4 + 8), name


def test_tcgen05_plans(lib):
    # tcgen05 kernel: 2048-token partitions (4096 for more than 16 heads), 128-token grain
    p = plan_for(lib, GB300_SMS, num_seqs=128, num_q_heads=32, num_kv_heads=8,
                 max_context_len=8192, dtype=B.PKV_BF16, kernel=3)
    assert (p.variant, p.split_tokens, p.num_splits) == (2, 2048, 4)
    p = plan_for(lib, GB300_SMS, num_seqs=256, num_q_heads=256, num_kv_heads=8,
                 max_context_len=8192, dtype=B.PKV_BF16, kernel=3)
    assert (p.variant, p.split_tokens, p.num_splits) == (2, 4096, 2)
    p = plan_for(lib, GB300_SMS, num_seqs=2, num_q_heads=8, num_kv_heads=2,
                 max_context_len=1000, kernel=3)
    assert p.variant == 2 and p.split_tokens % 128 == 0
    # a forced partition is rounded to the block size only (the kernel walks
    # it in 128-token groups, the last one ragged)
    for forced, want in ((80, 80), (208, 208), (70, 80)):
        p = plan_for(lib, GB300_SMS, num_seqs=2, num_q_heads=8, num_kv_heads=2,
                     max_context_len=1000, split_tokens=forced, kernel=3)
        assert (p.variant, p.split_tokens, p.num_splits) == (2, want, -(-1000 // want))


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=64, num_kv_heads=1), ERR_UNSUPPORTED),   # group of 64
    (dict(num_q_heads=8, num_kv_heads=2, kernel=1), ERR_UNSUPPORTED),  # CUDA cores, group 4
    (dict(head_dim=64, kernel=3), ERR_UNSUPPORTED),            # tcgen05 needs head_dim 128
    (dict(split_tokens=-1), ERR_INVALID),                       # no persistent schedule
    (dict(num_seqs=(1 << 26) + 1, num_q_heads=32, num_kv_heads=1,
          max_context_len=16), ERR_UNSUPPORTED),                # 2^31 + 32 output rows
    (dict(max_context_len=100, max_blocks_per_seq=4), ERR_INVALID),  # > MB * bs
])
def test_rejected_shapes(lib, kw, code):
    with pytest.raises(B.PkvError) as e:
        plan_for(lib, GB300_SMS, **kw)
    assert e.value.code == code


def test_bad_sm_count_and_null(lib):
    shape = B.make_shape(num_seqs=1, num_q_heads=1, num_kv_heads=1, head_dim=128, block_size=16,
                         num_blocks=4, max_blocks_per_seq=1, max_context_len=1)
    plan = B.Plan()
    assert lib.pkv_decode_plan_for(ctypes.byref(shape), 0, ctypes.byref(plan)) == ERR_INVALID
    assert lib.pkv_decode_plan_for(None, 152, ctypes.byref(plan)) == ERR_NULL
    assert lib.pkv_decode_plan_for(ctypes.byref(shape), 152, None) == ERR_NULL


# ------------------------------------------------------------ sweep
SWEEP = list(itertools.product(
    [1, 3, 16, 64, 257],                      # sequences
    [(8, 8), (32, 16), (32, 8), (64, 8), (128, 8), (256, 8)],   # (Hq, Hkv): groups 1-32
    [64, 128, 256],                           # head_dim
    [16, 32],                                 # block size
))


@pytest.mark.parametrize("sms", [8, 76, 152])
def test_partition_rule_sweep(lib, sms):
    """Every shape of the sweep, with automatic and forced partition sizes,
    plans exactly as the restated rule says, and the plan covers every token:
    (S-1)*P < max_context_len <= S*P, P a multiple of the block size."""
    rng = np.random.default_rng(sms)
    checked = 0
    for B_, (Hq, Hkv), D, bs in SWEEP:
        for maxL in (1, bs, int(rng.integers(2, 300)), 4096, int(rng.integers(300, 40000))):
            for split in (0, 0, int(rng.integers(1, 3000))):
                p = plan_for(lib, sms, num_seqs=B_, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D, block_size=bs, num_blocks=4096,
                             max_context_len=maxL, split_tokens=split)
                variant, P, S, grid, ws = expected_plan(B_, Hq, Hkv, D, bs, maxL, split, sms)
                got = (p.schedule, p.variant, p.split_tokens, p.num_splits, p.grid_ctas,
                       p.workspace_bytes)
                assert got == (0, variant, P, S, grid, ws), (B_, Hq, Hkv, D, bs, maxL, split)
                assert P % bs == 0 and (S - 1) * P < maxL <= S * P
                assert P <= MAX_BLOCKS_PER_CTA * bs or P == -(-maxL // bs) * bs
                assert p.warps_per_cta == warps(D, bs)
                assert p.stages_per_warp == stages(D, bs, heads_per_warp(variant, Hq // Hkv))
                checked += 1
    assert checked == len(SWEEP) * 15
