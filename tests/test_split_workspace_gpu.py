"""GPU tests of the split-KV workspace contract (through the C ABI).

With more than one partition per sequence, each partition's CTA leaves an
un-normalised partial (m, l, o) in the caller's workspace and the reduce
kernel merges them: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, the
cross-split rescale of the FlashAttention-style tiling (third page,
"FlashAttention deep integration").  These tests check from outside that
the workspace needs no initialisation, that one workspace serves calls whose
partition counts change, and that a bad block id in one partition disturbs
neither the other sequences nor the next call.

Tolerance: |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_268_gb300 import workloads as W
from parity import assert_close, device_inputs, widen_out

pytestmark = pytest.mark.gpu

MHA = W.scaled(W.WORKLOADS["llama7b_mha"], 6, 1300)                        # group 1
GQA = W.scaled(W.WORKLOADS["llama3_8b_gqa"], 8, 1500, min_len=16)          # group 4
CONT = W.scaled(W.WORKLOADS["cont_batch"], 16, 700)                        # group 4
LONG = W.scaled(W.WORKLOADS["long_ctx_gqa"], 2, 2600, lens="fixed")        # group 8, bs 32


def _decode(pkv, w, d, ws, split, out=None, lens=None, kernel=0):
    out = pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"] if lens is None else lens, w.scale, out,
                                max_context_len=w.max_context_len, split_tokens=split,
                                kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    return out


def _oracle(w, lens=None):
    return oracle.decode(W.bits(w.q), W.bits(w.k_cache), W.bits(w.v_cache), w.block_tables,
                         w.context_lens if lens is None else lens, w.scale, w.spec.dtype)


def _workspace(pkv, w, d, split, kernel=0):
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len, split,
                             kernel)
    assert pkv.decode_plan(shape).num_splits > 1
    return pkv.alloc_workspace(shape)


def _fill(ws: torch.Tensor, how: str, seed: int = 0):
    if how == "zeros":
        ws.zero_()
    elif how == "ones":                  # every float reads as NaN
        ws.fill_(0xFF)
    elif how == "random":
        g = torch.Generator(device="cpu").manual_seed(seed)
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, generator=g))
    else:
        raise ValueError(how)


@pytest.mark.parametrize("how", ["zeros", "ones", "random"])
@pytest.mark.parametrize("spec,split", [(MHA, 128), (GQA, 64), (CONT, 128), (LONG, 256)])
def test_workspace_needs_no_initialisation(pkv, spec, split, how):
    w = W.make(spec, seed=1)
    d = device_inputs(w)
    ws = _workspace(pkv, w, d, split)
    _fill(ws, how, seed=3)
    ref = _oracle(w)
    for rep in range(2):
        out = _decode(pkv, w, d, ws, split)
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), ref, f"{spec.name}/{how}/call {rep}")


@pytest.mark.parametrize("spec,split", [(MHA, 128), (GQA, 64), (CONT, 64), (LONG, 256)])
def test_split_counts_change_between_calls(pkv, spec, split):
    """One workspace over calls whose sequences change their partition count
    (fewer, more again, one partition, back; never past the table's blocks):
    every call matches the oracle."""
    w = W.make(spec, seed=2)
    d = device_inputs(w)
    ws = _workspace(pkv, w, d, split)
    base = w.context_lens.copy()
    variants = [base,
                np.maximum(1, base // 3).astype(np.int32),
                np.maximum(1, (base * 2) // 3).astype(np.int32),
                np.full_like(base, min(split, int(base.min()))),
                base]
    for i, lens in enumerate(variants):
        out = _decode(pkv, w, d, ws, split, lens=torch.from_numpy(lens).cuda())
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), _oracle(w, lens), f"{spec.name} call {i}")


@pytest.mark.parametrize("spec,split,kernel", [(GQA, 64, 0), (MHA, 128, 0), (LONG, 256, 0),
                                               (GQA, 256, 3)])
def test_bad_block_in_one_partition(pkv, spec, split, kernel):
    """A bad block id in the second partition of one sequence: the error word
    reads PKV_DEV_BAD_BLOCK_ID, the other sequences match the oracle (that
    sequence's rows are undefined), and the next call on the same workspace
    with a valid table is right everywhere."""
    w = W.make(spec, seed=0)
    d = device_inputs(w)
    ws = _workspace(pkv, w, d, split, kernel)
    bs = spec.block_size
    seq = int(np.argmax(w.context_lens))
    assert w.context_lens[seq] > split + bs
    j = split // bs                      # first block of the second partition
    good = int(d["block_tables"][seq, j])
    d["block_tables"][seq, j] = spec.num_blocks + 11
    out = _decode(pkv, w, d, ws, split, kernel=kernel)
    assert pkv.get_device_error() == 1
    ref = _oracle(w)
    others = [i for i in range(spec.num_seqs) if i != seq]
    assert_close(widen_out(out)[others], ref[others], "other sequences")
    d["block_tables"][seq, j] = good
    out = _decode(pkv, w, d, ws, split, kernel=kernel)
    assert pkv.get_device_error() == 0
    assert_close(widen_out(out), ref, "after the bad call")


def test_set_workspace_serves_calls_without_one(pkv):
    """pkv_set_workspace: a decode (and a fused step) given a NULL workspace
    uses the one set for the device; one too small is reported before any
    launch; host memory is refused; clearing it restores the error."""
    import ctypes
    lib = pkv.load_library()
    w = W.make(LONG, seed=6)
    d = device_inputs(w)
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len)
    need = pkv.decode_plan(shape).workspace_bytes
    assert need > 0
    ref = _oracle(w)
    big = torch.empty(need + 4096, dtype=torch.uint8, device="cuda")
    _fill(big, "ones")
    args = (ctypes.byref(shape), d["q"].data_ptr(), d["k_cache"].data_ptr(),
            d["v_cache"].data_ptr(), d["block_tables"].data_ptr(), d["context_lens"].data_ptr(),
            ctypes.c_float(w.scale))
    stream = torch.cuda.current_stream().cuda_stream
    try:
        assert lib.pkv_set_workspace(big.data_ptr(), need + 4096) == 0
        out = torch.full_like(d["q"], float("nan"))
        assert lib.pkv_paged_attn_decode(*args, out.data_ptr(), None, 0, stream) == 0
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), ref, "set workspace, C ABI")
        # the binding passes no workspace once one is set for the device
        pkv.set_workspace(big)
        n0 = pkv.launch_count()
        out2 = _decode(pkv, w, d, None, 0)
        assert pkv.launch_count() - n0 == 2
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
        # too small: rejected on the host, nothing launched
        small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
        assert lib.pkv_set_workspace(small.data_ptr(), need - 16) == 0
        n0 = pkv.launch_count()
        assert lib.pkv_paged_attn_decode(*args, out.data_ptr(), None, 0, stream) == -5
        assert pkv.launch_count() == n0
        # host memory is not a device workspace
        host = torch.empty(need, dtype=torch.uint8).pin_memory()
        assert lib.pkv_set_workspace(host.data_ptr(), need) == -2
    finally:
        pkv.set_workspace(None)
    assert lib.pkv_paged_attn_decode(*args, out.data_ptr(), None, 0, stream) == -5


@pytest.mark.parametrize("D,bs", [(64, 16), (128, 16), (256, 32)])
def test_reduce_builds_at_their_split_counts(pkv, D, bs):
    """The split reduce has three builds, chosen by the split count: two
    splits (the 40-register build; head_dim 256 uses the next one), up to
    the 64-register build's batch, and more.  Forced partition sizes put the
    longest sequence at each boundary; every row must match the oracle."""
    lens = np.array([1, bs, 2 * bs + 3, 300, 1200, 2000], dtype=np.int32)
    spec = W.WorkloadSpec("reduce", len(lens), 8, 2, D, bs, W.BF16, 0, 0, "uniform", (1, 1))
    spec = W.scaled(spec, len(lens), int(lens.max()))
    w = W.make(spec, seed=D + bs, lens=lens)
    d = device_inputs(w)
    ref = _oracle(w)
    Lmax = int(lens.max())
    for S in (2, 3, 8, 9, 16, 17, 33):
        split = -(-(-(-Lmax // S)) // bs) * bs          # partition size giving about S splits
        shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len, split)
        plan = pkv.decode_plan(shape)
        ws = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
        _fill(ws, "ones")
        out = _decode(pkv, w, d, ws, split)
        assert pkv.get_device_error() == 0
        assert_close(widen_out(out), ref, f"D={D} bs={bs} S={plan.num_splits}")


def test_set_workspace_serves_the_fused_step(pkv):
    """pkv_decode_step with a NULL workspace uses the set one, like the plain
    decode: same output and caches as with an explicit workspace."""
    w = W.make(GQA, seed=8)
    d = device_inputs(w)
    shape = pkv.decode_shape(d["q"], d["k_cache"], d["block_tables"], w.max_context_len)
    assert pkv.decode_plan(shape).workspace_bytes > 0
    k_new, v_new = w.k_new.cuda(), w.v_new.cuda()
    kc1, vc1 = d["k_cache"].clone(), d["v_cache"].clone()
    ref = pkv.decode_step(d["q"], k_new, v_new, kc1, vc1, d["block_tables"], d["context_lens"],
                          w.scale, max_context_len=w.max_context_len,
                          workspace=pkv.alloc_workspace(shape))
    big = pkv.alloc_workspace(shape)
    _fill(big, "random", 3)
    kc2, vc2 = d["k_cache"].clone(), d["v_cache"].clone()
    try:
        pkv.set_workspace(big)
        out = pkv.decode_step(d["q"], k_new, v_new, kc2, vc2, d["block_tables"], d["context_lens"],
                              w.scale, max_context_len=w.max_context_len)
        torch.cuda.synchronize()
    finally:
        pkv.set_workspace(None)
    assert pkv.get_device_error() == 0
    for a_, b_ in ((out, ref), (kc2, kc1), (vc2, vc1)):
        assert torch.equal(a_.view(torch.int16), b_.view(torch.int16))
