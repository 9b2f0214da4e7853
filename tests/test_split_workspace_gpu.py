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
