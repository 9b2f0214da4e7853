"""GPU parity of paged_attn_decode against the CPU oracle (through the C ABI).

Tolerance: |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise, the bound stated for
fp16/bf16 output with fp32 accumulation."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, gpu_decode, oracle_decode, widen_out

pytestmark = pytest.mark.gpu

# Oracle-sized versions of the five workloads: same heads, head_dim, block
# size, dtype and structure; fewer, shorter sequences spanning several tiles,
# several splits and a ragged last block.
SMALL = {
    "tiny_mha": W.WORKLOADS["tiny_mha"],
    "llama7b_mha": W.scaled(W.WORKLOADS["llama7b_mha"], 6, 1300),
    "llama3_8b_gqa": W.scaled(W.WORKLOADS["llama3_8b_gqa"], 8, 1500, min_len=16),
    "long_ctx_gqa": W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 2600, lens="fixed"),
    "cont_batch": W.scaled(W.WORKLOADS["cont_batch"], 16, 700),
}


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", W.ORDER)
def test_small_workloads(pkv, name, seed):
    w = W.make(SMALL[name], seed=seed)
    assert_close(widen_out(gpu_decode(pkv, w)), oracle_decode(w), f"{name}/{seed}")


def test_plan_selection(pkv):
    """split_tokens 0 lets the library choose the partition size, > 0 forces
    it; the tensor-core variant serves group sizes of 3 and more."""
    for name in W.ORDER:
        w = W.make(SMALL[name], seed=0)
        d = device_inputs(w)
        for split in (0, 64):
            plan = pkv.decode_plan(pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"],
                                                    w.max_context_len, split))
            assert plan.schedule == 0
            assert plan.variant == (0 if w.spec.group <= 2 else 1)
        assert plan.split_tokens == 64


def test_large_batch(pkv):
    """More than 2048 sequences of short contexts."""
    spec = W.scaled(W.WORKLOADS["llama3_8b_gqa"], 2100, 40)
    w = W.make(spec, seed=9)
    assert_close(widen_out(gpu_decode(pkv, w)), oracle_decode(w), "B=2100")


@pytest.mark.parametrize("split", [16, 64, 256, 512, 1 << 20])
def test_split_count_invariance(pkv, split):
    """Every partition size of the fixed-partition schedule gives the oracle's
    answer within tolerance (split_tokens > 0 selects that schedule)."""
    for name in ("llama7b_mha", "long_ctx_gqa"):
        w = W.make(SMALL[name], seed=5)
        assert_close(widen_out(gpu_decode(pkv, w, split_tokens=split)), oracle_decode(w),
                     f"{name}/split={split}")


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 6, 8, 12, 16, 24, 32])
@pytest.mark.parametrize("D,bs", [(64, 16), (128, 16), (128, 32), (256, 16), (64, 32), (256, 32)])
def test_shape_sweep(pkv, dtype, G, D, bs):
    Hkv = 2
    spec = W.WorkloadSpec("sweep", 5, G * Hkv, Hkv, D, bs, dtype, 0, 0, "uniform", (1, 1))
    lens = np.array([1, bs - 1, bs, bs + 1, 3 * bs + 5], dtype=np.int32)
    spec = W.scaled(spec, 5, int(lens.max()))
    w = W.make(spec, seed=G * 1000 + D + bs, lens=lens)
    for split in (0, bs, 2 * bs):   # auto partitions, one- and two-block partitions
        assert_close(widen_out(gpu_decode(pkv, w, split_tokens=split)), oracle_decode(w),
                     f"G={G} D={D} bs={bs} split={split}")


def test_edge_lengths(pkv):
    """ctx = 1, multiples of the block size and one either side, long tails,
    with automatic and forced partitions."""
    lens = np.array([1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1023, 1024, 1025], dtype=np.int32)
    for base in ("llama7b_mha", "llama3_8b_gqa", "long_ctx_gqa"):
        spec = W.scaled(W.WORKLOADS[base], len(lens), int(lens.max()))
        w = W.make(spec, seed=11, lens=lens)
        ref = oracle_decode(w)
        for split in (0, 512, 80):
            assert_close(widen_out(gpu_decode(pkv, w, split_tokens=split)), ref,
                         f"{base} split={split}")


@pytest.mark.parametrize("B", [1, 3, 37])
def test_few_blocks_and_single_long_sequence(pkv, B):
    """Batches with fewer KV blocks than warps in the grid, and a single
    long sequence that every CTA (or warp) takes a piece of."""
    rng = np.random.default_rng(B)
    lens = rng.integers(1, 40 if B > 1 else 20000, size=B).astype(np.int32)
    for base in ("llama7b_mha", "long_ctx_gqa"):
        spec = W.scaled(W.WORKLOADS[base], B, int(lens.max()))
        w = W.make(spec, seed=B, lens=lens)
        ref = oracle_decode(w)
        for split in (0, 48):
            assert_close(widen_out(gpu_decode(pkv, w, split_tokens=split)), ref,
                         f"{base} B={B} split={split}")


def test_all_context_one_returns_v(pkv):
    spec = W.scaled(W.WORKLOADS["llama3_8b_gqa"], 4, 1)
    w = W.make(spec, seed=2, lens=np.ones(4, dtype=np.int32))
    out = widen_out(gpu_decode(pkv, w))
    G = spec.group
    for i in range(4):
        p = w.block_tables[i, 0]
        v0 = w.v_cache[p, :, 0, :].double().cpu().numpy()
        for h in range(spec.num_q_heads):
            assert np.array_equal(out[i, h], v0[h // G])


def test_deterministic_and_shared_rows_identical(pkv):
    """Repeated calls are bit-identical; sequences with identical q, table and
    length give bit-identical rows (the shared-prefix sanity check)."""
    w = W.make(SMALL["cont_batch"], seed=3)
    d = device_inputs(w)
    d["q"][1] = d["q"][0]
    d["block_tables"][1] = d["block_tables"][0]
    d["context_lens"][1] = d["context_lens"][0]
    a = gpu_decode(pkv, w, d)
    b = gpu_decode(pkv, w, d)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a[0].view(torch.int16), a[1].view(torch.int16))


def test_bad_block_id_sets_device_error(pkv):
    """An out-of-range table entry is caught by the kernel's own range check:
    the unit is skipped and the error word reads PKV_DEV_BAD_BLOCK_ID."""
    w = W.make(SMALL["llama3_8b_gqa"], seed=0)
    d = device_inputs(w)
    d["block_tables"][2, 0] = w.spec.num_blocks + 7
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len)
    assert pkv.get_device_error() == 1
    assert pkv.get_device_error() == 0          # read clears it
    d["block_tables"][2, 0] = -3
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len)
    assert pkv.get_device_error() == 1


def test_bad_context_len_sets_device_error(pkv):
    w = W.make(SMALL["llama7b_mha"], seed=0)
    d = device_inputs(w)
    d["context_lens"][1] = 0
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len)
    assert pkv.get_device_error() == 2
    d["context_lens"][1] = w.max_context_len + 1
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len)
    assert pkv.get_device_error() == 2


def _sample_rows(w: W.Workload, n: int, rng) -> np.ndarray:
    B, Hq = w.spec.num_seqs, w.spec.num_q_heads
    n = min(n, B * Hq)
    longest = int(np.argmax(w.context_lens))
    shortest = int(np.argmin(w.context_lens))
    rows = {(longest, 0), (longest, Hq - 1), (shortest, Hq // 2), (B - 1, Hq - 1)}
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(Hq))))
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("name", W.ORDER)
def test_full_size_sampled(pkv, name):
    """Full-size workloads in the benchmark's launch configuration (and with
    1024-token partitions forced); the oracle recomputes a sample of
    (sequence, head) rows one by one."""
    w = W.make(name, seed=0, device="cuda")
    d = device_inputs(w)
    rows = _sample_rows(w, 48, np.random.default_rng(0))
    ref = oracle.decode_rows(rows, W.bits(w.q), W.bits(w.k_cache), W.bits(w.v_cache),
                             w.block_tables, w.context_lens, w.scale, w.spec.dtype)
    for split in (0, 1024):
        out = widen_out(gpu_decode(pkv, w, d, split_tokens=split))
        assert np.all(np.isfinite(out))
        assert_close(out[rows[:, 0], rows[:, 1]], ref, f"{name} split={split}")


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("G", [1, 4, 8, 12, 16, 24, 32])
@pytest.mark.parametrize("bs", [16, 32])
def test_tcgen05_kernel(pkv, dtype, G, bs):
    """The tcgen05/TMEM kernel (kernel=3) on ragged lengths spanning several
    128-token groups and partitions, including forced partitions that are not
    a multiple of 128 tokens (80 and 208: every partition ends in a ragged
    group)."""
    Hkv = 2
    spec = W.WorkloadSpec("tc", 6, G * Hkv, Hkv, 128, bs, dtype, 0, 0, "uniform", (1, 1))
    lens = np.array([1, 127, 128, 129, 700, 1500], dtype=np.int32)
    spec = W.scaled(spec, 6, int(lens.max()))
    w = W.make(spec, seed=G * 7 + bs, lens=lens)
    d = device_inputs(w)
    plan = pkv.decode_plan(pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"],
                                            w.max_context_len, 0, 3))
    assert plan.variant == 2 and plan.schedule == 0
    ref = oracle_decode(w)
    for split in (0, 256, 1 << 20, 80, 208):
        if split in (80, 208):
            sp = pkv.decode_plan(pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"],
                                                  w.max_context_len, split, 3))
            assert sp.split_tokens == -(-split // bs) * bs     # rounded to the block size only
        out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], w.scale, max_context_len=w.max_context_len,
                                    split_tokens=split, kernel=3)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), ref, f"tcgen05 G={G} bs={bs} split={split}")


def test_kernel_choice_rules(pkv):
    w = W.make(W.scaled(W.WORKLOADS["llama3_8b_gqa"], 2, 64), seed=0)
    d = device_inputs(w)
    shp = lambda k, split=0: pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"],
                                              w.max_context_len, split, k)
    assert pkv.decode_plan(shp(0)).variant == 1          # group 4 -> mma.sync
    assert pkv.decode_plan(shp(3)).variant == 2
    with pytest.raises(pkv.PkvError):
        pkv.decode_plan(shp(1))                          # CUDA cores need group <= 2
    with pytest.raises(pkv.PkvError):
        pkv.decode_plan(shp(3, -1))                      # negative partition sizes


@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("G", [8, 32])
def test_rising_logits_rescale(pkv, kernel, G):
    """K rows scaled up along each sequence make the logits keep growing, so
    the running maxima rise again and again: the rescale of the partial
    output (in registers for mma.sync, in TMEM for tcgen05) runs many times
    within one partition."""
    Hkv, bs = 2, 16
    spec = W.WorkloadSpec("ramp", 3, G * Hkv, Hkv, 128, bs, W.BF16, 0, 0, "uniform", (1, 1))
    lens = np.array([700, 1300, 2100], dtype=np.int32)
    spec = W.scaled(spec, 3, int(lens.max()))
    w = W.make(spec, seed=17 + G, lens=lens)
    for i, L in enumerate(lens):
        t = np.arange(int(L))
        f = torch.from_numpy((1.0 + t / 96.0).astype(np.float32)).to(torch.bfloat16)
        blocks = torch.from_numpy(w.block_tables[i, t // bs].astype(np.int64))
        offs = torch.from_numpy((t % bs).astype(np.int64))
        rows = w.k_cache[blocks, :, offs, :]                   # [L, Hkv, D]
        w.k_cache[blocks, :, offs, :] = (rows.float() * f.float()[:, None, None]).to(torch.bfloat16)
    d = device_inputs(w)
    ref = oracle_decode(w)
    for split in (0, 1 << 20):
        out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], w.scale, max_context_len=w.max_context_len,
                                    split_tokens=split, kernel=kernel)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), ref, f"rising logits kernel={kernel} G={G} split={split}")


def test_tcgen05_bad_block_id(pkv):
    """The tcgen05 kernel's range check: the unit is skipped, the error word is
    set, TMEM is released (the next call on the same GPU runs normally)."""
    w = W.make(SMALL["long_ctx_gqa"], seed=2)
    d = device_inputs(w)
    d["block_tables"][1, 3] = w.spec.num_blocks + 5
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], w.scale, max_context_len=w.max_context_len, kernel=3)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 1
    d["block_tables"][1, 3] = int(w.block_tables[1, 3])
    out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], w.scale, max_context_len=w.max_context_len,
                                kernel=3)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert_close(widen_out(out), oracle_decode(w), "tcgen05 after a bad block id")


def test_wait_timeout_is_reported_and_gpu_stays_usable(pkv):
    """Failure detection without a GPU fault: a warp waits on an mbarrier that
    nothing arrives on, with the kernels' bounded wait; the wait runs out, the
    host reads PKV_DEV_TIMEOUT, and the next decode on the same context is
    correct."""
    import time
    t0 = time.time()
    pkv.selftest_wait_timeout(20_000)
    assert pkv.get_device_error() == 4
    assert time.time() - t0 < 5.0
    assert pkv.get_device_error() == 0        # read clears it
    w = W.make(SMALL["llama3_8b_gqa"], seed=4)
    assert_close(widen_out(gpu_decode(pkv, w)), oracle_decode(w), "decode after a timeout")
    with pytest.raises(pkv.PkvError):
        pkv.selftest_wait_timeout(0)
