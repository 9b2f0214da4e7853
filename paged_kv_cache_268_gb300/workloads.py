"""Seeded synthetic decode batches shaped like the paged-KV serving workloads.

This module only *makes inputs*: context lengths, block tables, slot mappings
and N(0, 1) values rounded to fp16/bf16.  It holds none of the attention or
append arithmetic, and it is the one module shared by the CUDA path's callers
(tests, benchmark) and the oracle's callers (tests, CPU baseline).

Recipe (the pages name no public benchmark or dataset, so these synthetic
batches stand in for "long and short requests mixed in production", third
page, "PagedAttention" and "continuous batching" sections):

* lengths: per workload, see ``WORKLOADS`` (fixed, uniform, log-normal).
* block tables: a seeded permutation of the physical pool [0, NB) is handed out
  consecutively (sequence 0 logical blocks 0..n0-1, then sequence 1, ...), so
  the physical blocks of a sequence are scattered over the pool.  Table entries
  past ceil(L / bs) are -1 (never read by a correct kernel).
* prefix sharing (continuous-batching workload only): sequences 8k..8k+7 form a
  group; logical blocks j < min(32, (L-1) // bs) (the full blocks of the first
  512 tokens that precede the block receiving the new token) map to the group's
  shared physical blocks, so one set of K/V data serves all eight, and no
  appended token ever lands in a shared block.
* values: q, new k/v rows and both caches ~ N(0, 1) in float32, rounded to the
  element type (round-to-nearest-even, torch's conversion).  In the long
  context workload every K row (token, kv head) is first multiplied by
  u ~ U(0.5, 2) to spread the logits.  Pool blocks that no table references
  are filled with a NaN pattern so that a stray read shows up in the output.
* the appended token of each sequence sits at position L - 1 (context_lens
  counts it), slot = table[i][(L-1) // bs] * bs + (L-1) % bs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

F16, BF16 = 0, 1
_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}
# quiet-NaN patterns used to poison unreferenced pool blocks
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: int
    num_blocks: int          # physical pool size NB
    max_blocks_per_seq: int  # MB, row stride of the block table
    lens: str                # "fixed", "uniform", "lognormal"
    len_args: tuple = ()
    scale: float = 0.0       # 0 -> 1/sqrt(head_dim) as float32
    share_prefix: bool = False
    k_row_spread: bool = False

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        s = self.scale if self.scale else 1.0 / math.sqrt(self.head_dim)
        return float(np.float32(s))


WORKLOADS = {
    # tiny MHA decode: 4 seqs, 8 heads, D=64, bs=16, lens {1,17,64,200}, fp16,
    # scale 1/8, table = random permutation of a 64-block pool
    "tiny_mha": WorkloadSpec("tiny_mha", 4, 8, 8, 64, 16, F16, 64, 13,
                             "fixed", (1, 17, 64, 200), scale=0.125),
    # Llama-7B-shaped MHA decode: 64 seqs, 32/32 heads, D=128, bs=16, fp16,
    # lens U{512..4096}, 16384-block pool
    "llama7b_mha": WorkloadSpec("llama7b_mha", 64, 32, 32, 128, 16, F16, 16384,
                                256, "uniform", (512, 4096)),
    # Llama-3-8B-shaped GQA decode: 128 seqs, 32/8 heads, bf16, lens log-normal
    # (median 1024, sigma 1.0), clipped to [16, 8192]
    "llama3_8b_gqa": WorkloadSpec("llama3_8b_gqa", 128, 32, 8, 128, 16, BF16,
                                  65536, 512, "lognormal", (1024, 1.0, 16, 8192)),
    # long-context low-batch GQA decode: 4 seqs of 32768 tokens, 64/8 heads,
    # bs=32, bf16, K rows scaled by U(0.5, 2)
    "long_ctx_gqa": WorkloadSpec("long_ctx_gqa", 4, 64, 8, 128, 32, BF16, 8192,
                                 1024, "fixed", (32768,) * 4, k_row_spread=True),
    # continuous-batching step: 256 seqs, 32/8 heads, bs=16, fp16, lens
    # U{1..2048} (after the append), 512-token prefixes shared by groups of 8
    "cont_batch": WorkloadSpec("cont_batch", 256, 32, 8, 128, 16, F16, 32768,
                               128, "uniform", (1, 2048), share_prefix=True),
    # not one of the five workloads: a wide-group batch (16 query heads per kv
    # head) for comparing the tensor-core kernels
    "wide_gqa16": WorkloadSpec("wide_gqa16", 64, 128, 8, 128, 16, BF16, 16384, 256,
                               "uniform", (512, 4096)),
    "wide_gqa32": WorkloadSpec("wide_gqa32", 64, 256, 8, 128, 16, BF16, 16384, 256,
                               "uniform", (512, 4096)),
}
ORDER = ["tiny_mha", "llama7b_mha", "llama3_8b_gqa", "long_ctx_gqa", "cont_batch"]


def scaled(spec: WorkloadSpec, num_seqs: int, max_len: int,
           min_len: int = 1, lens: str = "uniform", name: str | None = None) -> WorkloadSpec:
    """Same heads, head_dim, block size and dtype, fewer and shorter sequences
    (for cases the oracle finishes in seconds)."""
    mb = -(-max_len // spec.block_size)
    nb = max(64, int(num_seqs * mb * 1.25) + 8)
    largs = (min_len, max_len) if lens == "uniform" else (max_len,) * num_seqs
    return replace(spec, name=name or f"{spec.name}_x{num_seqs}_{max_len}",
                   num_seqs=num_seqs, num_blocks=nb, max_blocks_per_seq=mb,
                   lens=lens, len_args=largs)


def context_lengths(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    B = spec.num_seqs
    if spec.lens == "fixed":
        lens = np.asarray(spec.len_args, dtype=np.int64)
        assert lens.shape == (B,)
    elif spec.lens == "uniform":
        lo, hi = spec.len_args
        lens = rng.integers(lo, hi + 1, size=B)
    elif spec.lens == "lognormal":
        median, sigma, lo, hi = spec.len_args
        lens = np.clip(np.rint(np.exp(rng.normal(math.log(median), sigma, size=B))), lo, hi)
    else:
        raise ValueError(spec.lens)
    lens = lens.astype(np.int32)
    assert lens.min() >= 1 and lens.max() <= spec.max_blocks_per_seq * spec.block_size
    return lens


def block_tables(spec: WorkloadSpec, lens: np.ndarray, rng: np.random.Generator):
    """Return (tables [B, MB] int32 with -1 past each sequence's last block,
    used [NB] bool)."""
    B, bs, MB, NB = spec.num_seqs, spec.block_size, spec.max_blocks_per_seq, spec.num_blocks
    perm = rng.permutation(NB).astype(np.int32)
    nxt = 0

    def take(n):
        nonlocal nxt
        if nxt + n > NB:
            raise ValueError(f"pool of {NB} blocks too small")
        ids = perm[nxt:nxt + n]
        nxt += n
        return ids

    tables = np.full((B, MB), -1, dtype=np.int32)
    nblk = -(-lens // bs)
    if spec.share_prefix:
        nshared = np.minimum(32, (lens - 1) // bs)
        for g0 in range(0, B, 8):
            grp = slice(g0, min(g0 + 8, B))
            shared = take(int(nshared[grp].max()))
            for i in range(grp.start, grp.stop):
                ns = int(nshared[i])
                tables[i, :ns] = shared[:ns]
                tables[i, ns:nblk[i]] = take(int(nblk[i]) - ns)
    else:
        for i in range(B):
            tables[i, :nblk[i]] = take(int(nblk[i]))
    used = np.zeros(NB, dtype=bool)
    for i in range(B):
        used[tables[i, :nblk[i]]] = True
    return tables, used


def append_slots(spec: WorkloadSpec, lens: np.ndarray, tables: np.ndarray) -> np.ndarray:
    """Slot of the token at position L-1 of every sequence (this step's new token)."""
    pos = lens.astype(np.int64) - 1
    blk = tables[np.arange(spec.num_seqs), pos // spec.block_size].astype(np.int64)
    return (blk * spec.block_size + pos % spec.block_size).astype(np.int32)


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    context_lens: np.ndarray     # [B] int32
    block_tables: np.ndarray     # [B, MB] int32
    slot_mapping: np.ndarray     # [B] int32
    used_blocks: np.ndarray      # [NB] bool
    q: torch.Tensor              # [B, Hq, D]
    k_new: torch.Tensor          # [B, Hkv, D]
    v_new: torch.Tensor          # [B, Hkv, D]
    k_cache: torch.Tensor        # [NB, Hkv, bs, D]
    v_cache: torch.Tensor        # [NB, Hkv, bs, D]
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return self.spec.softmax_scale

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max())

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode call reads: sum_i L_i * Hkv * D * 2 * 2."""
        s = self.spec
        return int(self.context_lens.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2 * 2

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct cache rows one call touches (a shared
        prefix block is counted once)."""
        s = self.spec
        rows_of = {}
        for i in range(s.num_seqs):
            L = int(self.context_lens[i])
            for j in range(-(-L // s.block_size)):
                p = int(self.block_tables[i, j])
                rows = min(s.block_size, L - j * s.block_size)
                rows_of[p] = max(rows_of.get(p, 0), rows)
        return sum(rows_of.values()) * s.num_kv_heads * s.head_dim * 2 * 2


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _gen(device, seed: int, stream: int):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) % (2 ** 63))
    return g


def make(spec: WorkloadSpec | str, seed: int = 0, device: str | torch.device = "cpu",
         lens: np.ndarray | None = None) -> Workload:
    """Build one seeded batch.  Small tensors are drawn on the CPU; the two
    caches are drawn on ``device`` (use the GPU for the full-size pools)."""
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    device = torch.device(device)
    rng = np.random.default_rng([seed, ORDER.index(spec.name) if spec.name in ORDER else 99])
    if lens is None:
        lens = context_lengths(spec, rng)
    else:
        lens = np.asarray(lens, dtype=np.int32)
        spec = replace(spec, num_seqs=int(lens.shape[0]))
        assert lens.min() >= 1 and lens.max() <= spec.max_blocks_per_seq * spec.block_size
    tables, used = block_tables(spec, lens, rng)
    slots = append_slots(spec, lens, tables)
    tdt = _TORCH_DTYPE[spec.dtype]
    B, Hq, Hkv, D = spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    gcpu = _gen("cpu", seed, 1)
    q = _normal((B, Hq, D), gcpu, "cpu").to(tdt).to(device)
    k_new = _normal((B, Hkv, D), gcpu, "cpu").to(tdt).to(device)
    v_new = _normal((B, Hkv, D), gcpu, "cpu").to(tdt).to(device)
    cshape = (spec.num_blocks, Hkv, spec.block_size, D)
    gk = _gen(device, seed, 2)
    kf = _normal(cshape, gk, device)
    if spec.k_row_spread:
        u = torch.rand(cshape[:-1] + (1,), generator=gk, device=device, dtype=torch.float32)
        kf.mul_(u.mul_(1.5).add_(0.5))
    k_cache = kf.to(tdt)
    del kf
    gv = _gen(device, seed, 3)
    v_cache = _normal(cshape, gv, device).to(tdt)
    unused = torch.from_numpy(np.nonzero(~used)[0]).to(device=device, dtype=torch.long)
    if unused.numel():
        nan = NAN_BITS[spec.dtype]
        for c in (k_cache, v_cache):
            c.view(torch.int16).index_fill_(0, unused, nan)
    return Workload(spec, seed, lens, tables, slots, used, q, k_new, v_new,
                    k_cache, v_cache)


def bits(t) -> np.ndarray:
    """Host copy of a 16-bit tensor as its raw element patterns (uint16);
    uint16 numpy arrays pass through unchanged."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return t
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
