// Paged decode attention on the 5th-generation tensor cores (tcgen05, TMEM),
// for wide query groups.  Same contract, grid and split-KV partials as
// paged_decode_kernel (one CTA per (sequence, kv head, partition)); only the
// inner loop differs.  The method is the same FlashAttention-style pass over
// the paged cache (third page, "PagedAttention" and "FlashAttention"
// sections) of softmax(q . K^T * scale) . V (second page, section 3.1).
//
// The partition is walked in groups of 128 tokens (128 / bs blocks):
//   * TMA lands the group's K and V as 32 KB tiles (two 128-byte-swizzled
//     column boxes of 128 rows) in a ring of three tile slots, in the order
//     K0 V0 K1 V1 ...; a slot is refilled as soon as the MMA reading it has
//     completed.
//   * One thread issues S^T[128 tok x N] = K . Q^T (tcgen05.mma, M = 128,
//     both operands K-major in shared memory, accumulator in TMEM).
//   * Each thread owns one token row of S^T (tcgen05.ld 32x32b): logits in
//     log2 units, masked past the context end.  The group's per-head maxima
//     go through shared memory; the running maxima m are raised only when a
//     group exceeds them by more than 2^8 (then O and the sums are rescaled
//     in TMEM), so P = 2^(s - m) stays below 256.  P^T goes to shared memory
//     as a K-major operand (bfloat16 as a hi + lo pair, binary16 as is).
//   * One thread issues O^T[128 d x N] += V^T . P^T (V^T read MN-major from
//     the same V tile).
// At the end every thread holds one output dimension d of every head.
#pragma once

#include "pkv_decode.cuh"

namespace pkv {

// Shared-memory layout of the tcgen05 kernel (N = padded group size).
template <int N>
struct TcLayout {
  static constexpr int TILE = 32768;            // 128 tokens x 128 dims x 2 B
  static constexpr int SLOTS = 3;
  static constexpr int Q_BYTES = 2 * N * 128;   // Q^T: 2 column boxes x N rows x 128 B
  static constexpr int P_BYTES = 2 * N * 128;   // P^T: 2 token chunks x N rows x 128 B
  static constexpr int OFF_Q = SLOTS * TILE;
  static constexpr int OFF_P = OFF_Q + Q_BYTES;              // hi, then lo
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;        // 3 slot + qk + pv barriers
  static constexpr int OFF_RED = OFF_BAR + 64;               // [4 warps][N] floats
  static constexpr int OFF_MISC = OFF_RED + 4 * N * 4;       // TMEM address, then m per head
  static constexpr int OFF_IDS = OFF_MISC + 16 + N * 4;
  static constexpr int BYTES = OFF_IDS + kMaxBlocksPerCta * 4 + 1024;
  static constexpr int TMEM_COLS = 2 * N < 32 ? 32 : 2 * N;  // S^T then O^T
};

template <bool BF, int BS, int N>
__global__ void __launch_bounds__(128, 1)
    paged_decode_tc(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  constexpr int D = 128;
  using LY = TcLayout<N>;
  constexpr int GB = 128 / BS;   // blocks per group
  static_assert(N % 16 == 0 && N <= 32, "N is 16 or 32");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_slot0 = sb + LY::OFF_BAR;               // slot s at + 8 s
  const uint32_t bar_qk = sb + LY::OFF_BAR + 24;
  const uint32_t bar_pv = sb + LY::OFF_BAR + 32;
  float* red = reinterpret_cast<float*>(smem + LY::OFF_RED);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::OFF_MISC);
  float* mshare = reinterpret_cast<float*>(smem + LY::OFF_MISC + 16);
  int* ids = reinterpret_cast<int*>(smem + LY::OFF_IDS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  int idx = blockIdx.x;
  const int split = idx % a.S;
  idx /= a.S;
  const int kvh = idx % a.Hkv;
  const int seq = idx / a.Hkv;
  const int L = a.context_lens[seq];
  if (L < 1 || L > a.max_ctx) {
    if (tid == 0 && split == 0 && kvh == 0) record_error(a.err, kDevBadContext);
    return;
  }
  const int t0 = split * a.P;
  if (t0 >= L) return;
  const int t1 = min(t0 + a.P, L);
  const int j0 = t0 / BS;
  const int nblk = (t1 - t0 + BS - 1) / BS;
  const int ngroups = (t1 - t0 + 127) / 128;
  const size_t row0 = (size_t)seq * a.Hq + (size_t)kvh * a.G;

  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  bool bad = false;
  for (int k = tid; k < nblk; k += 128) {
    const int p = __ldg(a.block_tables + (size_t)seq * a.MB + j0 + k);
    bad |= (p < 0) | (p >= a.NB);
    ids[k] = p;
  }
  if (tid < 5) mbar_init(bar_slot0 + 8 * tid, 1);
  // Q^T operand, K-major 128-byte swizzle: column box c (dims 64c..64c+63),
  // row n (head), 16-byte chunk cc at position cc ^ (n % 8); heads >= G are 0.
  for (int i = tid; i < 2 * N * 8; i += 128) {
    const int c = i / (N * 8), rem = i - c * (N * 8), n = rem >> 3, cc = rem & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < a.G) v = *reinterpret_cast<const uint4*>(a.q + (row0 + n) * D + c * 64 + cc * 8);
    const uint32_t dst = sb + LY::OFF_Q + c * (N * 128) + n * 128 + ((cc ^ (n & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), LY::TMEM_COLS);
  if (tid == 0) fence_mbar_init();
  tc_fence_before();
  const bool any_bad = __syncthreads_or(bad);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (any_bad) {
    if (tid == 0) record_error(a.err, kDevBadBlock);
    if (warp == 0) tmem_dealloc(tmem, LY::TMEM_COLS);
    return;
  }
  const uint32_t tS = tmem, tO = tmem + N;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  // Tile t: K of group t/2 (t even) or V (t odd), into slot t % 3.
  auto issue_tile = [&](int t) {
    const int g = t >> 1, slot = t % 3;
    const int b0 = g * GB, nb = min(GB, nblk - b0);
    const uint32_t bar = bar_slot0 + 8 * slot;
    const CUtensorMap* map = (t & 1) ? &tmV : &tmK;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb * BS * 256));
    for (int b = 0; b < nb; ++b) {
      const int y = (ids[b0 + b] * a.Hkv + kvh) * BS;
      const uint32_t dst = sb + slot * LY::TILE + b * BS * 128;
      tma_load_2d(dst, map, 0, y, bar);
      tma_load_2d(dst + 16384, map, 64, y, bar);
    }
  };
  if (tid == 0) {
    issue_tile(0);
    issue_tile(1);
    if (ngroups > 1) issue_tile(2);
  }

  const uint32_t idesc_qk = umma_idesc_f16(BF, 0, 0, N, 128);
  const uint32_t idesc_pv = umma_idesc_f16(BF, 1, 0, N, 128);
  float mref[N], lth[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    mref[n] = -INFINITY;
    lth[n] = 0.f;
  }
  bool fail = false;

  for (int g = 0; g < ngroups; ++g) {
    const int tK = 2 * g, tV = 2 * g + 1;
    const uint32_t kslot = sb + (tK % 3) * LY::TILE, vslot = sb + (tV % 3) * LY::TILE;
    // S^T = K . Q^T
    if (tid == 0) {
      fail |= !mbar_wait(bar_slot0 + 8 * (tK % 3), (tK / 3) & 1);
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = umma_desc_sw128(kslot + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t bd =
            umma_desc_sw128(sb + LY::OFF_Q + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
        umma_f16(tS, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
      }
      umma_commit(bar_qk);
    }
    fail |= !mbar_wait(bar_qk, g & 1);
    tc_fence_after();
    if (tid == 0 && g + 1 < ngroups) issue_tile(2 * g + 3);  // V of g+1 into K(g)'s slot

    // this thread's token row of S^T
    float x[N];
#pragma unroll
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tmem_ld16(tS + lane_off + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) x[c + i] = v[i];
    }
    const int rows = min(128, t1 - (t0 + g * 128));  // valid tokens of this group
    const bool valid = tid < rows;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      x[n] = valid ? x[n] * a.scale_log2 : -INFINITY;
      float v = x[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
      if (lane == 0) red[warp * N + n] = v;
    }
    __syncthreads();
    float gmax[N];
    bool rescale = false;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      gmax[n] = fmaxf(fmaxf(red[n], red[N + n]), fmaxf(red[2 * N + n], red[3 * N + n]));
      rescale |= gmax[n] > mref[n] + 8.f;
    }
    if (g > 0) {
      // PV of g-1 done: P, O and the V(g-1) slot are free again
      fail |= !mbar_wait(bar_pv, (g - 1) & 1);
      tc_fence_after();
      if (tid == 0 && g + 1 < ngroups) issue_tile(2 * g + 2);  // K of g+1
    }
    if (rescale) {
      float alpha[N];
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float mn = fmaxf(mref[n], gmax[n]);
        alpha[n] = fast_exp2(mref[n] - mn);
        mref[n] = mn;
        lth[n] *= alpha[n];
      }
      if (g > 0) {
#pragma unroll
        for (int c = 0; c < N; c += 16) {
          float v[16];
          tmem_ld16(tO + lane_off + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= alpha[c + i];
          tmem_st16(tO + lane_off + c, v);
        }
      }
    }
    // P^T operand: row n (head), token tid in chunk tid / 64
    {
      const int chunk = tid >> 6, t = tid & 63;
      const uint32_t pbase = sb + LY::OFF_P + chunk * (N * 128) + (t & 7) * 2;
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float p = fast_exp2(x[n] - mref[n]);
        lth[n] += p;
        const uint32_t addr = pbase + n * 128 + ((((t >> 3) ^ (n & 7))) << 4);
        const uint16_t hi = to_elem<BF>(p);
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(hi) : "memory");
        if constexpr (BF) {
          const float hf = __uint_as_float(static_cast<uint32_t>(hi) << 16);
          const uint16_t lo = to_elem<BF>(p - hf);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr + LY::P_BYTES), "h"(lo) : "memory");
        }
      }
    }
    if (rows < 128) {
      // Last, ragged group: V rows past the context end (and blocks never
      // loaded) may hold anything; P is 0 there but 0 * NaN is not, so clear
      // them once the tile has landed.
      fail |= !mbar_wait(bar_slot0 + 8 * (tV % 3), (tV / 3) & 1);
      for (int i = tid; i < (128 - rows) * 16; i += 128) {
        const int r = rows + (i >> 4), c = i & 15;
        const uint32_t addr = vslot + (c >> 3) * 16384 + r * 128 + (c & 7) * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // O^T += V^T . P^T
    if (tid == 0) {
      tc_fence_after();
      fail |= !mbar_wait(bar_slot0 + 8 * (tV % 3), (tV / 3) & 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = umma_desc_sw128(vslot + kk * 2048, 16384, 1024);
        const uint64_t bd =
            umma_desc_sw128(sb + LY::OFF_P + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
        umma_f16(tO, ad, bd, idesc_pv, (g > 0 || kk > 0) ? 1u : 0u);
      }
      if constexpr (BF) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = umma_desc_sw128(vslot + kk * 2048, 16384, 1024);
          const uint64_t bd = umma_desc_sw128(
              sb + LY::OFF_P + LY::P_BYTES + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
          umma_f16(tO, ad, bd, idesc_pv, 1u);
        }
      }
      umma_commit(bar_pv);
    }
  }

  // Epilogue: this thread's output dimension d = tid for every head.
  fail |= !mbar_wait(bar_pv, (ngroups - 1) & 1);
  tc_fence_after();
  float o[N];
#pragma unroll
  for (int c = 0; c < N; c += 16) {
    float v[16];
    tmem_ld16(tO + lane_off + c, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) o[c + i] = v[i];
  }
#pragma unroll
  for (int n = 0; n < N; ++n) {
    float v = lth[n];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    if (lane == 0) red[warp * N + n] = v;
  }
  if (tid == 0) {
#pragma unroll
    for (int n = 0; n < N; ++n) mshare[n] = mref[n];
  }
  __syncthreads();
  const bool single = (L + a.P - 1) / a.P == 1;
  const int d = tid;
#pragma unroll
  for (int n = 0; n < N; ++n) {
    if (n < a.G) {
      const float lsum = red[n] + red[N + n] + red[2 * N + n] + red[3 * N + n];
      if (single) {
        a.out[(row0 + n) * D + d] = to_elem<BF>(o[n] / lsum);
      } else {
        const size_t pr = (row0 + n) * a.S + split;
        a.part_o[pr * D + d] = o[n];
        if (d == 0) a.part_ml[pr] = make_float2(mshare[n], lsum);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, LY::TMEM_COLS);
  if (fail && tid == 0) record_error(a.err, kDevTimeout);
}

}  // namespace pkv
