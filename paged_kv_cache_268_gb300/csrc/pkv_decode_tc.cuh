// Paged decode attention on the 5th-generation tensor cores (tcgen05, TMEM),
// warp-specialised, for wide query groups.  Same contract, grid and split-KV
// partials as paged_decode_kernel (one CTA per (sequence, kv head,
// partition)); only the inner loop differs.  The method is the same
// FlashAttention-style pass over the paged cache (third page,
// "PagedAttention" and "FlashAttention" sections) of
// softmax(q . K^T * scale) . V (second page, section 3.1).
//
// The partition is walked in groups of 128 tokens (128 / bs blocks).  The
// warps split the work and hand it on through mbarriers, so loads, tensor
// core work and softmax of different groups overlap:
//   * warp SW (one lane), producer: TMA lands each group's K and V as 32 KB
//     tiles (two 128-byte-swizzled column boxes of 128 rows) in a ring of
//     SLOTS tile slots, K one group ahead of V (K0 K1 V0 K2 V1 ... V(n-1)),
//     the order the MMA consumes them in; a slot is refilled as soon as the
//     MMA reading it has completed.
//   * warp SW + 1 (one lane), MMA issuer: S^T[128 tok x N] = K . Q^T into one
//     of two TMEM buffers (both operands K-major in shared memory), and,
//     once the softmax warps have published P of a group,
//     O^T[128 d x N] += V^T . P^T (V^T read MN-major from the V tile),
//     issuing whichever is ready first.  So QK of group g runs on the tensor
//     pipe while group g-1 is in softmax.
//   * warps 0..SW-1, softmax (SW = 4 for N = 16, 8 for N = 32): a thread owns
//     token row t of S^T (TMEM lane t, tcgen05.ld 32x32b) for 16 heads (warps
//     w and w + 4 share a lane quarter and split the heads): logits in log2
//     units, masked past the context end.  The running per-head maxima m are
//     raised only when a group exceeds them by more than 2^8, detected with
//     one barrier reduction per group; then O and the partial sums are
//     rescaled in TMEM.
//     P = 2^(s - m) (so P < 256) goes to shared memory as a K-major operand
//     (bfloat16 as a hi + lo pair, binary16 as is); with N = 32 it alternates
//     between two buffers, so the softmax of group g + 1 does not wait for
//     the PV of group g.
// At the end a softmax thread holds output dimension d = t of its 16 heads.
// Fused append (k_new set): the CTA whose partition holds position L-1
// writes this step's K/V row to its cache slot and, once the tiles holding
// it have landed, the MMA thread writes it into them before the MMAs read
// them.
// Every wait is bounded; on a timeout each role stops, loads still in flight
// get a bounded wait, TMEM is freed and the device error word is set.
#pragma once

#include "pkv_decode.cuh"

namespace pkv {

// Shared-memory layout of the tcgen05 kernel (N = padded group size).
template <int N>
struct TcLayout {
  static constexpr int SOFT_WARPS = N > 16 ? 8 : 4;  // 16 heads per softmax thread
  static constexpr int HPT = N * 4 / SOFT_WARPS;
  static constexpr int THREADS = (SOFT_WARPS + 2) * 32;
  static constexpr int TILE = 32768;            // 128 tokens x 128 dims x 2 B
  // N = 16 fits two CTAs per SM with three slots each; N = 32 one CTA with five
  static constexpr int SLOTS = N > 16 ? 5 : 3;
  static constexpr int Q_BYTES = 2 * N * 128;   // Q^T: 2 column boxes x N rows x 128 B
  static constexpr int P_BYTES = 2 * N * 128;   // P^T: 2 token chunks x N rows x 128 B
  static constexpr int PBUF = N > 16 ? 2 : 1;   // P buffers (hi + lo each)
  static constexpr int OFF_Q = SLOTS * TILE;
  static constexpr int OFF_P = OFF_Q + Q_BYTES;              // buffer i: hi, then lo
  // barriers: full[SLOTS], empty[SLOTS], s_full[2], s_free[2], p_full[PBUF],
  // pv_done[PBUF]
  static constexpr int B_FULL = 0, B_EMPTY = SLOTS, B_SFULL = 2 * SLOTS,
                       B_SFREE = 2 * SLOTS + 2, B_PFULL = 2 * SLOTS + 4,
                       B_PVDONE = 2 * SLOTS + 4 + PBUF, NBAR = 2 * SLOTS + 4 + 2 * PBUF;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES * PBUF;
  static constexpr int OFF_RED = OFF_BAR + ((NBAR * 8 + 15) & ~15);  // [4 warps][N] floats
  static constexpr int OFF_MISC = OFF_RED + 4 * N * 4;        // TMEM address
  static constexpr int OFF_IDS = OFF_MISC + 16;
  static constexpr int OFF_NEW = OFF_IDS + kMaxBlocksPerCta * 4;  // fused append: new K, V rows
  static constexpr int BYTES = OFF_NEW + 2 * 128 * 2 + 1024;
  static constexpr int TMEM_COLS = 3 * N <= 64 ? 64 : 128;    // S0, S1, O
};

template <bool BF, int BS, int N>
__global__ void __launch_bounds__(TcLayout<N>::THREADS, N > 16 ? 1 : 2)
    paged_decode_tc(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
  constexpr int D = 128;
  using LY = TcLayout<N>;
  constexpr int SL = LY::SLOTS;
  constexpr int GB = 128 / BS;   // blocks per group
  constexpr int SOFT = LY::SOFT_WARPS * 32;   // softmax threads, named barrier 1
  constexpr int HPT = LY::HPT;                 // heads per softmax thread
  static_assert(N % 16 == 0 && N <= 32, "N is 16 or 32");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + LY::OFF_BAR + 8 * i; };
  float* red = reinterpret_cast<float*>(smem + LY::OFF_RED);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::OFF_MISC);
  int* ids = reinterpret_cast<int*>(smem + LY::OFF_IDS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int idx = blockIdx.x;
  const int split = idx % a.S;
  idx /= a.S;
  const int kvh = idx % a.Hkv;
  const int seq = idx / a.Hkv;
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // launched as a programmatic dependent of the previous kernel on the
  // stream: no memory is touched before that kernel has finished, and the
  // reduce (which reads the lengths before its own wait) may launch only
  // after that
  pdl_wait();
  pdl_launch_dependents();
  // block ids and length, as in paged_decode_kernel
  const int t0 = split * a.P;
  const int j0 = t0 / BS;
  const int32_t* trow = a.block_tables + (size_t)seq * a.MB + j0;
  const int L = a.context_lens[seq];
  if (split == 0)
    for (int k = tid; k < min(a.P / BS, a.MB - j0); k += LY::THREADS) ids[k] = __ldg(trow + k);
  if (L < 1 || L > a.max_ctx) {
    if (tid == 0 && split == 0 && kvh == 0) record_error(a.err, kDevBadContext);
    return;
  }
  if (t0 >= L) return;
  const int t1 = min(t0 + a.P, L);
  const int nblk = (t1 - t0 + BS - 1) / BS;
  const int ngroups = (t1 - t0 + 127) / 128;
  const size_t row0 = (size_t)seq * a.Hq + (size_t)kvh * a.G;

  bool bad = false;
  for (int k = tid; k < nblk; k += LY::THREADS) {
    const int p = split == 0 ? ids[k] : __ldg(trow + k);
    bad |= (p < 0) | (p >= a.NB);
    ids[k] = p;
  }
  if (tid < LY::NBAR) {
    const bool many = (tid >= LY::B_SFREE && tid < LY::B_SFREE + 2) ||
                      (tid >= LY::B_PFULL && tid < LY::B_PFULL + LY::PBUF);
    mbar_init(bar(tid), many ? SOFT : 1);
  }
  // Q^T operand, K-major 128-byte swizzle: column box c (dims 64c..64c+63),
  // row n (head), 16-byte chunk cc at position cc ^ (n % 8); heads >= G are 0.
  for (int i = tid; i < 2 * N * 8; i += LY::THREADS) {
    const int c = i / (N * 8), rem = i - c * (N * 8), n = rem >> 3, cc = rem & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < a.G) v = *reinterpret_cast<const uint4*>(a.q + (row0 + n) * D + c * 64 + cc * 8);
    const uint32_t dst = sb + LY::OFF_Q + c * (N * 128) + n * 128 + ((cc ^ (n & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
  }
  // fused append: position L-1 is in this partition
  const bool fused = a.k_new != nullptr && L - 1 >= t0 && L - 1 < t1;
  if (fused) {
    for (int c = tid; c < 2 * (D / 8); c += LY::THREADS) {
      const bool isv = c >= D / 8;
      const int gc = isv ? c - D / 8 : c;
      const uint4 x = *reinterpret_cast<const uint4*>((isv ? a.v_new : a.k_new) +
                                                      ((size_t)seq * a.Hkv + kvh) * D + gc * 8);
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sb + LY::OFF_NEW + c * 16),
                   "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w)
                   : "memory");
    }
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
  if (fused && tid < 2 * (D / 8)) {
    // the new row to its cache slot (the ids are in range past the check)
    const int jb = (L - 1) / BS, r = (L - 1) - jb * BS;
    const size_t dst = (((size_t)ids[jb - j0] * a.Hkv + kvh) * BS + r) * D;
    const bool isv = tid >= D / 8;
    const int gc = isv ? tid - D / 8 : tid;
    uint4 x;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                 : "r"(sb + LY::OFF_NEW + tid * 16));
    *reinterpret_cast<uint4*>((isv ? a.v_cache : a.k_cache) + dst + gc * 8) = x;
  }
  const uint32_t tO = tmem + 2 * N;   // S buffer b at tmem + b * N
  bool fail = false;
  // ring order: K(g) is tile tile_k(g), V(g) is tile tile_v(g)
  auto tile_k = [&](int g) { return g == 0 ? 0 : 2 * g - 1; };
  auto tile_v = [&](int g) { return g + 1 < ngroups ? 2 * g + 2 : 2 * ngroups - 1; };

  if (warp == LY::SOFT_WARPS) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();   // the KV stream is read once
      const int ntiles = 2 * ngroups;
      int t = 0;
      for (; t < ntiles; ++t) {
        const int slot = t % SL;
        if (t >= SL && !mbar_wait(bar(LY::B_EMPTY + slot), ((t / SL) - 1) & 1)) {
          fail = true;
          break;
        }
        // tile t: K of group (t + 1) / 2 (t odd, or 0), else V of t / 2 - 1;
        // the last tile is V of the last group
        const bool is_v = t == ntiles - 1 ? ngroups > 0 : (t > 0 && (t & 1) == 0);
        const int g = t == ntiles - 1 ? ngroups - 1 : (is_v ? t / 2 - 1 : (t + 1) / 2);
        const int b0 = g * GB, nb = min(GB, nblk - b0);
        const uint32_t full = bar(LY::B_FULL + slot);
        const CUtensorMap* map = is_v ? &tmV : &tmK;
        mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * BS * 256));
        for (int b = 0; b < nb; ++b) {
          const int y = (ids[b0 + b] * a.Hkv + kvh) * BS;
          const uint32_t dst = sb + slot * LY::TILE + b * BS * 128;
          tma_load_2d(dst, map, 0, y, full, policy);
          tma_load_2d(dst + 16384, map, 64, y, full, policy);
        }
      }
      // every slot's last issued load lands before the CTA may exit (the
      // earlier ones were consumed, so they landed)
      for (int tt = max(0, t - SL); tt < t; ++tt)
        mbar_wait(bar(LY::B_FULL + tt % SL), (tt / SL) & 1, 100000000ull);
    }
  } else if (warp == LY::SOFT_WARPS + 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_f16(BF, 0, 0, N, 128);
      const uint32_t idesc_pv = umma_idesc_f16(BF, 1, 0, N, 128);
      // Two streams of work, each in group order: S(gs) once K(gs) has landed
      // and S buffer gs % 2 is free again (the softmax of gs - 2 read it),
      // and PV(gp) once the softmax has published P(gp) and V(gp) has landed.
      // Whichever is ready goes first, so a late K tile never holds back a
      // PV (and the V slot it frees).  S stays at most one group ahead of PV
      // (gs <= gp + 1): then the tile a slot held before the one tested has
      // always landed, so a barrier is never tested one phase early, where
      // its parity would alias.  Gives up after 0.5 s without progress.
      auto s_ready = [&](int g) {
        const int tK = tile_k(g);
        return mbar_test_wait(bar(LY::B_FULL + tK % SL), (tK / SL) & 1) &&
               (g < 2 || mbar_test_wait(bar(LY::B_SFREE + (g & 1)), ((g - 2) >> 1) & 1));
      };
      auto pv_ready = [&](int j) {
        const int tV = tile_v(j);
        return mbar_test_wait(bar(LY::B_PFULL + j % LY::PBUF), (j / LY::PBUF) & 1) &&
               mbar_test_wait(bar(LY::B_FULL + tV % SL), (tV / SL) & 1);
      };
      // fused append: group and tile row of position L-1
      const int g_new = fused ? ((L - 1) - t0) / 128 : -1;
      const int r_new = ((L - 1) - t0) & 127;
      auto patch = [&](uint32_t tile, int isv) {
#pragma unroll
        for (int gc = 0; gc < D / 8; ++gc) {
          uint4 x;
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
                       : "r"(sb + LY::OFF_NEW + (isv * (D / 8) + gc) * 16));
          const uint32_t dst =
              tile + (gc >> 3) * 16384 + r_new * 128 + (((gc & 7) ^ (r_new & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(x.x), "r"(x.y),
                       "r"(x.z), "r"(x.w)
                       : "memory");
        }
        fence_proxy_async_smem();
      };
      auto issue_s = [&](int g) {
        const int tK = tile_k(g), ks = tK % SL, b = g & 1;
        const uint32_t kslot = sb + ks * LY::TILE;
        if (g == g_new) patch(kslot, 0);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = umma_desc_sw128(kslot + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd =
              umma_desc_sw128(sb + LY::OFF_Q + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + b * N, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(LY::B_SFULL + b));
        umma_commit(bar(LY::B_EMPTY + ks));    // K slot free
      };
      auto issue_pv = [&](int j) {
        const int tV = tile_v(j), vs = tV % SL, pb = j % LY::PBUF;
        const uint32_t pbuf = sb + LY::OFF_P + pb * 2 * LY::P_BYTES;
        const uint32_t vslot = sb + vs * LY::TILE;
        if (j == g_new) patch(vslot, 1);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = umma_desc_sw128(vslot + kk * 2048, 16384, 1024);
          const uint64_t bd =
              umma_desc_sw128(pbuf + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
          umma_f16(tO, ad, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if constexpr (BF) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_desc_sw128(vslot + kk * 2048, 16384, 1024);
            const uint64_t bd = umma_desc_sw128(
                pbuf + LY::P_BYTES + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024);
            umma_f16(tO, ad, bd, idesc_pv, 1u);
          }
        }
        umma_commit(bar(LY::B_PVDONE + pb));   // O updated, P buffer pb free
        umma_commit(bar(LY::B_EMPTY + vs));    // V slot free
      };
      int gs = 0, gp = 0, idle = 0;
      bool fresh = true;       // progress since the clock was last read
      uint64_t t_last = 0;
      while (gp < ngroups) {
        bool moved = false;
        if (gs < ngroups && gs <= gp + 1 && s_ready(gs)) {
          issue_s(gs++);
          moved = true;
        }
        if (gp < gs && pv_ready(gp)) {
          issue_pv(gp++);
          moved = true;
        }
        if (moved) {
          fresh = true;
          idle = 0;
          continue;
        }
        if (++idle < 256) continue;
        idle = 0;
        const uint64_t now = globaltimer_ns();
        if (fresh) {
          t_last = now;
          fresh = false;
        } else if (now - t_last > 500000000ull) {
          break;
        }
      }
      fail = gp < ngroups;
    }
  } else {
    // ---------------------------------------------------------- softmax
    // The 128 softmax threads meet at named barriers, so none of them leaves
    // the loop early: after a failed wait a thread skips its later waits and
    // runs on with whatever is there; the error word reports it.
    const int tok = tid & 127;               // token row = TMEM lane
    const int quarter = warp & 3;
    const int h0 = (warp >> 2) * HPT;       // first head of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float m[HPT], lth[HPT];
#pragma unroll
    for (int n = 0; n < HPT; ++n) {
      m[n] = -INFINITY;
      lth[n] = 0.f;
    }
    auto wait = [&](uint32_t bar_addr, uint32_t parity) {
      if (!fail && !mbar_wait(bar_addr, parity)) fail = true;
    };
    for (int g = 0; g < ngroups; ++g) {
      const int b = g & 1;
      wait(bar(LY::B_SFULL + b), (g >> 1) & 1);
      __syncwarp();
      tc_fence_after();
      float x[HPT];
#pragma unroll
      for (int c = 0; c < HPT; c += 16) {
        float v[16];
        tmem_ld16(tmem + b * N + lane_off + h0 + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[c + i] = v[i];
      }
      tc_fence_before();
      mbar_arrive(bar(LY::B_SFREE + b));
      const int rows = min(128, t1 - (t0 + g * 128));  // valid tokens of this group
      const bool valid = tok < rows;
      bool up = false;
#pragma unroll
      for (int n = 0; n < HPT; ++n) {
        x[n] = valid ? x[n] * a.scale_log2 : -INFINITY;
        up |= x[n] > m[n] + 8.f;
      }
      // one barrier per group: does any token push a maximum up by 2^8?
      if (named_bar_or(1, SOFT, up)) {
        float gmax[HPT];
#pragma unroll
        for (int n = 0; n < HPT; ++n) {
          float v = x[n];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
          if (lane == 0) red[quarter * N + h0 + n] = v;
        }
        named_bar_sync(1, SOFT);
#pragma unroll
        for (int n = 0; n < HPT; ++n) {
          const float* r = red + h0 + n;
          gmax[n] = fmaxf(fmaxf(r[0], r[N]), fmaxf(r[2 * N], r[3 * N]));
        }
        float alpha[HPT];
#pragma unroll
        for (int n = 0; n < HPT; ++n) {
          const float mn = fmaxf(m[n], gmax[n]);
          alpha[n] = fast_exp2(m[n] - mn);
          m[n] = mn;
          lth[n] *= alpha[n];
        }
        if (g > 0) {
          // O holds groups 0..g-1 once the PV of g-1 has completed
          wait(bar(LY::B_PVDONE + (g - 1) % LY::PBUF), ((g - 1) / LY::PBUF) & 1);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < HPT; c += 16) {
            float v[16];
            tmem_ld16(tO + lane_off + h0 + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha[c + i];
            tmem_st16(tO + lane_off + h0 + c, v);
          }
        }
        // red is next written after the next group's barrier
      }
      // P buffer g % PBUF is free once the PV of g - PBUF has completed
      const int pb = g % LY::PBUF;
      if (g >= LY::PBUF) wait(bar(LY::B_PVDONE + pb), ((g - LY::PBUF) / LY::PBUF) & 1);
      {
        // P^T operand: row h (head), token tok in chunk tok / 64
        const int chunk = tok >> 6, t = tok & 63;
        const uint32_t pbase =
            sb + LY::OFF_P + pb * 2 * LY::P_BYTES + chunk * (N * 128) + (t & 7) * 2;
#pragma unroll
        for (int n = 0; n < HPT; ++n) {
          const float p = fast_exp2(x[n] - m[n]);
          lth[n] += p;
          const int h = h0 + n;
          const uint32_t addr = pbase + h * 128 + (((t >> 3) ^ (h & 7)) << 4);
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
        const int tV = tile_v(g);
        wait(bar(LY::B_FULL + tV % SL), (tV / SL) & 1);
        const uint32_t vslot = sb + (tV % SL) * LY::TILE;
        for (int i = tid; i < (128 - rows) * 16; i += SOFT) {
          const int r = rows + (i >> 4), c = i & 15;
          const uint32_t addr = vslot + (c >> 3) * 16384 + r * 128 + (c & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(LY::B_PFULL + pb));
    }

    // Epilogue: this thread's output dimension d = tok for its heads.
    wait(bar(LY::B_PVDONE + (ngroups - 1) % LY::PBUF), ((ngroups - 1) / LY::PBUF) & 1);
    __syncwarp();
    tc_fence_after();
    float o[HPT];
#pragma unroll
    for (int c = 0; c < HPT; c += 16) {
      float v[16];
      tmem_ld16(tO + lane_off + h0 + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) o[c + i] = v[i];
    }
    named_bar_sync(1, SOFT);   // every thread is past its last use of red
#pragma unroll
    for (int n = 0; n < HPT; ++n) {
      float v = lth[n];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      if (lane == 0) red[quarter * N + h0 + n] = v;
    }
    named_bar_sync(1, SOFT);
    const bool single = (L + a.P - 1) / a.P == 1;
    const int d = tok;
#pragma unroll
    for (int n = 0; n < HPT; ++n) {
      const int h = h0 + n;
      if (h < a.G) {
        const float* r = red + h;
        const float lsum = r[0] + r[N] + r[2 * N] + r[3 * N];
        if (single) {
          a.out[(row0 + h) * D + d] = to_elem<BF>(o[n] / lsum);
        } else {
          const size_t pr = (row0 + h) * a.S + split;
          a.part_o[pr * D + d] = o[n];
          if (d == 0) a.part_ml[pr] = make_float2(m[n], lsum);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, LY::TMEM_COLS);
  if (fail) record_error(a.err, kDevTimeout);
}

}  // namespace pkv
