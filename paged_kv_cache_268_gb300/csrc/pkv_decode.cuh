// Paged single-token decode attention kernels for sm_103a.
//
// One CTA handles one (sequence, kv head, split) unit: the tokens
// [split * P, min((split + 1) * P, L)) of one sequence, for every query head of
// the kv head's group.  The method is the paged attention of the third page
// ("PagedAttention": fixed-size physical blocks, a block table, indirect
// addressing) computed FlashAttention-style (third page, "FlashAttention deep
// integration": tile the KV, keep partial results on chip, one pass over HBM),
// with the plain definition softmax(q . K^T * scale) . V of the second page,
// section 3.1.
//
// Data path, per warp (each warp owns an independent pipeline):
//   block-table gather  -> the CTA copies its partition's physical block ids
//                          into shared memory once (and range-checks them)
//   stage K/V blocks    -> lane 0 issues TMA tiled loads of whole [bs, D] K and
//                          V tiles (contiguous 2-8 KB each in the
//                          [NB, Hkv, bs, D] cache) into a ring of NS stages,
//                          completing on per-stage mbarriers, 128-byte
//                          swizzled so that the fragment reads below are
//                          bank-conflict free, marked evict-first in L2
//                          (each K/V row is read once per step)
//   QK + online softmax -> FP32 logits in log2 units, running max m and sum l
//   PV accumulate       -> FP32 output accumulators rescaled by 2^(m_old-m_new)
// The warps of a CTA then merge their (m, l, o) in shared memory; the CTA
// writes the normalised output (one split) or its partial (m, l, o) for the
// cross-split reduce kernel.
//
// Two compute variants share that pipeline:
//   SIMT (group size 1-2): CUDA cores.  Lane (t8 = lane % 8, quarter = lane / 8)
//     dots token t8 of an 8-row pass with its quarter of q; two xor-shuffles
//     finish each dot, three more give the block max.  For PV each lane owns
//     D / 32 output dims.
//   MMA (group size 3-32): the group's query heads form the N = 8 sides of
//     NT = ceil(G / 8) mma.sync.m16n8k16 tiles.  S^T[16 tok x 8 heads] = K_tile . Q^T (K via
//     ldmatrix, Q^T fragments held in registers), P^T is transposed in
//     registers with movmatrix into the B operand of O^T[16 d x 8 heads] +=
//     V^T . P^T (V via ldmatrix.trans), so a head's column of S^T, P^T and O^T
//     always lives in the same thread.  With bfloat16 inputs P goes in as a
//     hi + lo pair of bfloat16 values.
#pragma once

#include "pkv_geometry.h"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

// Byte offset of 16-byte chunk `gc` (0 .. D/8-1) of row `r` in a [BS, D] tile
// stored as D/64 column boxes of BS rows x 128 bytes with the 128-byte swizzle
// (chunk c of row r sits at chunk position c ^ (r % 8)).
template <int BS>
__device__ __forceinline__ uint32_t tile_off(int r, int gc) {
  return static_cast<uint32_t>((gc >> 3) * BS * 128 + r * 128 + (((gc & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ SIMT
template <bool BF, int D, int BS, int GH>
struct SimtCompute {
  static constexpr int QPL = D / 4;    // q values per lane (its quarter of D)
  static constexpr int CPQ = D / 32;   // 16-byte chunks per quarter
  static constexpr int OPL = D / 32;   // output dims per lane
  static constexpr int PASSES = BS / 8;
  static constexpr int NH = GH;        // heads this warp produces

  float q[GH][QPL];
  float o[GH][OPL];
  float m[GH], l[GH];

  // q rows of the group start at `qg` (GH rows of D elements); each lane keeps
  // its quarter of every row in FP32.
  __device__ __forceinline__ void load_q(const uint16_t* qg, int /*G*/, int lane) {
    const int dq = lane >> 3;
#pragma unroll
    for (int gh = 0; gh < GH; ++gh) {
      const uint16_t* qrow = qg + gh * D + dq * QPL;
#pragma unroll
      for (int i = 0; i < QPL; i += 8) {
        uint4 u = *reinterpret_cast<const uint4*>(qrow + i);
        float2 f0 = unpack2<BF>(u.x), f1 = unpack2<BF>(u.y), f2 = unpack2<BF>(u.z),
               f3 = unpack2<BF>(u.w);
        q[gh][i + 0] = f0.x; q[gh][i + 1] = f0.y; q[gh][i + 2] = f1.x; q[gh][i + 3] = f1.y;
        q[gh][i + 4] = f2.x; q[gh][i + 5] = f2.y; q[gh][i + 6] = f3.x; q[gh][i + 7] = f3.y;
      }
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int gh = 0; gh < GH; ++gh) {
#pragma unroll
      for (int e = 0; e < OPL; ++e) o[gh][e] = 0.f;
      m[gh] = -INFINITY;
      l[gh] = 0.f;
    }
  }

  __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, float scale_log2,
                                        int lane) {
    const int t8 = lane & 7, dq = lane >> 3;
    float s[PASSES][GH];
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      const int r = ps * 8 + t8;
      float acc[GH];
#pragma unroll
      for (int gh = 0; gh < GH; ++gh) acc[gh] = 0.f;
#pragma unroll
      for (int i = 0; i < CPQ; ++i) {
        uint32_t x0, x1, x2, x3;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                     : "r"(kt + tile_off<BS>(r, dq * CPQ + i)));
        const float2 f0 = unpack2<BF>(x0), f1 = unpack2<BF>(x1), f2 = unpack2<BF>(x2),
                     f3 = unpack2<BF>(x3);
#pragma unroll
        for (int gh = 0; gh < GH; ++gh) {
          const float* qq = &q[gh][i * 8];
          acc[gh] = fmaf(qq[0], f0.x, acc[gh]); acc[gh] = fmaf(qq[1], f0.y, acc[gh]);
          acc[gh] = fmaf(qq[2], f1.x, acc[gh]); acc[gh] = fmaf(qq[3], f1.y, acc[gh]);
          acc[gh] = fmaf(qq[4], f2.x, acc[gh]); acc[gh] = fmaf(qq[5], f2.y, acc[gh]);
          acc[gh] = fmaf(qq[6], f3.x, acc[gh]); acc[gh] = fmaf(qq[7], f3.y, acc[gh]);
        }
      }
#pragma unroll
      for (int gh = 0; gh < GH; ++gh) {
        float v = acc[gh];
        v += __shfl_xor_sync(kFull, v, 8);
        v += __shfl_xor_sync(kFull, v, 16);
        s[ps][gh] = (r < valid) ? v * scale_log2 : -INFINITY;
      }
    }
    float p[PASSES][GH];
#pragma unroll
    for (int gh = 0; gh < GH; ++gh) {
      float mx = s[0][gh];
#pragma unroll
      for (int ps = 1; ps < PASSES; ++ps) mx = fmaxf(mx, s[ps][gh]);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
      const float mn = fmaxf(m[gh], mx);
      const float alpha = fast_exp2(m[gh] - mn);
      m[gh] = mn;
      float ls = 0.f;
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        p[ps][gh] = fast_exp2(s[ps][gh] - mn);
        ls += p[ps][gh];
      }
      l[gh] = l[gh] * alpha + ls;
#pragma unroll
      for (int e = 0; e < OPL; ++e) o[gh][e] *= alpha;
    }
    // PV: lane owns dims [lane * OPL, lane * OPL + OPL)
    constexpr int BYTES = OPL * 2;                  // 4, 8 or 16 bytes per lane per row
    const int gc = (lane * BYTES) >> 4;
    const int within = (lane * BYTES) & 15;
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int r = ps * 8 + t;
        if (r < valid) {
          const uint32_t addr = vt + tile_off<BS>(r, gc) + within;
          float vf[OPL];
          if constexpr (OPL == 2) {
            uint32_t x0;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x0) : "r"(addr));
            const float2 f0 = unpack2<BF>(x0);
            vf[0] = f0.x; vf[1] = f0.y;
          } else if constexpr (OPL == 4) {
            uint32_t x0, x1;
            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(x0), "=r"(x1) : "r"(addr));
            const float2 f0 = unpack2<BF>(x0), f1 = unpack2<BF>(x1);
            vf[0] = f0.x; vf[1] = f0.y; vf[2] = f1.x; vf[3] = f1.y;
          } else {
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(addr));
            const float2 f0 = unpack2<BF>(x0), f1 = unpack2<BF>(x1), f2 = unpack2<BF>(x2),
                         f3 = unpack2<BF>(x3);
            vf[0] = f0.x; vf[1] = f0.y; vf[2] = f1.x; vf[3] = f1.y;
            vf[4] = f2.x; vf[5] = f2.y; vf[6] = f3.x; vf[7] = f3.y;
          }
#pragma unroll
          for (int gh = 0; gh < GH; ++gh) {
            const float pt = __shfl_sync(kFull, p[ps][gh], t);
#pragma unroll
            for (int e = 0; e < OPL; ++e) o[gh][e] = fmaf(pt, vf[e], o[gh][e]);
          }
        }
      }
    }
  }

  // Leave each head's (m, l, o) for the CTA merge.
  __device__ __forceinline__ void publish(float* cm, float* cl, float* co, int lane) {
#pragma unroll
    for (int gh = 0; gh < GH; ++gh) {
      float lt = l[gh];
      lt += __shfl_xor_sync(kFull, lt, 1);
      lt += __shfl_xor_sync(kFull, lt, 2);
      lt += __shfl_xor_sync(kFull, lt, 4);
      if (lane == 0) { cm[gh] = m[gh]; cl[gh] = lt; }
#pragma unroll
      for (int e = 0; e < OPL; ++e) co[gh * D + lane * OPL + e] = o[gh][e];
    }
  }
};

// ------------------------------------------------------------------ MMA
// NT n-tiles of 8 query heads each (group sizes up to 8 * NT).
template <bool BF, int D, int BS, int NT = 1>
struct MmaCompute {
  static constexpr int KS = D / 16;    // k-steps of QK, d-tiles of PV
  static constexpr int MT = BS / 16;   // 16-token m-tiles per block
  static constexpr int NH = 8 * NT;    // heads this warp produces (N of the tiles)

  uint32_t qf[KS][NT][2];              // Q^T B-fragments
  float o[KS][NT][4];                  // O^T accumulators
  float m[NT][2], l[NT][2];            // heads nt*8 + 2*(lane%4) + {0, 1}

  // q rows of the group start at `qg` (G rows of D elements); lane holds the
  // Q^T B-fragments of heads nt*8 + lane/4 (zero for the padding heads >= G).
  __device__ __forceinline__ void load_q(const uint16_t* qg, int G, int lane) {
    const int c = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + (lane >> 2);
      const bool real = h < G;
      const uint16_t* qrow = qg + (real ? h : 0) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][nt][0] = real ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + c) : 0u;
        qf[ks][nt][1] = real ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + c) : 0u;
      }
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[ks][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
    }
  }

  __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, float scale_log2,
                                        int lane) {
    float s[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
      const int r = mt * 16 + (lane & 15);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(kt + tile_off<BS>(r, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_16816<BF>(s[mt][nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
      }
    }
    // logits in log2 units; rows past the context end are masked
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = mt * 16 + (lane >> 2) + ((e >> 1) << 3);
          const float x = (tok < valid) ? s[mt][nt][e] * scale_log2 : -INFINITY;
          s[mt][nt][e] = x;
          mx[e & 1] = fmaxf(mx[e & 1], x);
        }
      float alpha[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = mx[j];
        v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
        v = fmaxf(v, __shfl_xor_sync(kFull, v, 8));
        v = fmaxf(v, __shfl_xor_sync(kFull, v, 16));
        const float mn = fmaxf(m[nt][j], v);
        alpha[j] = fast_exp2(m[nt][j] - mn);
        m[nt][j] = mn;
        l[nt][j] *= alpha[j];
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pe = fast_exp2(s[mt][nt][e] - m[nt][e & 1]);
          s[mt][nt][e] = pe;
          l[nt][e & 1] += pe;
        }
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][nt][e] *= alpha[e & 1];
    }

    if (valid < BS) {
      // Rows past the context end carry whatever the block held; P is 0 there,
      // but 0 * NaN would still poison the MMA, so clear those V rows.
      constexpr int ROWB = 128;
      const int nz = (BS - valid) * (D / 64) * (ROWB / 16);  // 16-byte stores
      for (int i = lane; i < nz; i += 32) {
        const int per_box = (BS - valid) * (ROWB / 16);
        const int box = i / per_box, rem = i % per_box;
        const int r = valid + rem / (ROWB / 16), c = rem % (ROWB / 16);
        const uint32_t addr = vt + box * BS * ROWB + r * ROWB + c * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
      }
      __syncwarp();
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // P^T as the B operand.  bfloat16 keeps only 8 significant bits, so P
      // is carried as hi + lo (both bfloat16, ~16 bits together) and
      // multiplied twice; binary16's 11 bits are enough on their own.
      uint32_t b0[NT], b1[NT], c0[NT], c1[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t h0 = pack2<BF>(s[mt][nt][0], s[mt][nt][1]);
        const uint32_t h1 = pack2<BF>(s[mt][nt][2], s[mt][nt][3]);
        b0[nt] = movmatrix_trans(h0);
        b1[nt] = movmatrix_trans(h1);
        c0[nt] = c1[nt] = 0;
        if constexpr (BF) {
          const float2 f0 = unpack2<BF>(h0), f1 = unpack2<BF>(h1);
          c0[nt] = movmatrix_trans(pack2<BF>(s[mt][nt][0] - f0.x, s[mt][nt][1] - f0.y));
          c1[nt] = movmatrix_trans(pack2<BF>(s[mt][nt][2] - f1.x, s[mt][nt][3] - f1.y));
        }
      }
      const int r = mt * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int dt = 0; dt < KS; ++dt) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(vt + tile_off<BS>(r, 2 * dt + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816<BF>(o[dt][nt], a0, a1, a2, a3, b0[nt], b1[nt]);
          if constexpr (BF) mma_16816<BF>(o[dt][nt], a0, a1, a2, a3, c0[nt], c1[nt]);
        }
      }
    }
  }

  __device__ __forceinline__ void publish(float* cm, float* cl, float* co, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float lt = l[nt][j];
        lt += __shfl_xor_sync(kFull, lt, 4);
        lt += __shfl_xor_sync(kFull, lt, 8);
        lt += __shfl_xor_sync(kFull, lt, 16);
        if (lane < 4) { cm[nt * 8 + 2 * lane + j] = m[nt][j]; cl[nt * 8 + 2 * lane + j] = lt; }
      }
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = dt * 16 + (lane >> 2) + ((e >> 1) << 3);
          const int h = nt * 8 + 2 * (lane & 3) + (e & 1);
          co[h * D + d] = o[dt][nt][e];
        }
    }
  }
};

// ------------------------------------------------------------------ kernel
template <bool BF, int D, int BS, int NW, int NS, class Compute>
__global__ void __launch_bounds__(NW * 32, 1)
    paged_decode_kernel(const __grid_constant__ DecodeArgs a,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  constexpr int TILE = BS * D * 2;
  constexpr int STAGE = 2 * TILE;
  constexpr int NH = Compute::NH;
  // The warps' final (m, l, o) merge reuses the ring; barriers and block ids
  // sit after whichever of the two is larger.
  constexpr int RING = NW * NS * STAGE;
  constexpr int MERGE = NW * NH * (D + 2) * 4;
  constexpr int TAIL = ((RING > MERGE ? RING : MERGE) + 15) & ~15;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TAIL);
  int* ids = reinterpret_cast<int*>(bars + NW * NS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int idx = blockIdx.x;
  const int split = idx % a.S;
  idx /= a.S;
  const int kvh = idx % a.Hkv;
  const int seq = idx / a.Hkv;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // The grid is launched as a programmatic dependent of the previous kernel
  // on the stream (the last step's reduce): it may become resident while that
  // kernel finishes, and touches no memory before it has.  Only then may the
  // reduce start launching (it reads the lengths before its own wait, so
  // everything before this grid must be complete); it waits for this grid's
  // completion before reading partials.
  pdl_wait();
  pdl_launch_dependents();

  // Block-table gather for this partition (indirect addressing), range-
  // checked.  The first partition of a sequence is never empty, so it loads
  // its block ids while the context length is in flight (one round trip for
  // both); the others load them once the length shows they are not empty (an
  // empty CTA then exits after a single load).  split < S keeps j0 inside the
  // row: t0 < max_context_len <= MB * bs.
  const int t0 = split * a.P;
  const int j0 = t0 / BS;
  const int32_t* trow = a.block_tables + (size_t)seq * a.MB + j0;
  const int L = a.context_lens[seq];
  if (split == 0)
    for (int k = threadIdx.x; k < min(a.P / BS, a.MB - j0); k += NW * 32) ids[k] = __ldg(trow + k);
  if (L < 1 || L > a.max_ctx) {
    if (threadIdx.x == 0 && split == 0 && kvh == 0) record_error(a.err, kDevBadContext);
    return;
  }
  if (t0 >= L) return;
  const int t1 = min(t0 + a.P, L);
  const int nblk = (t1 - t0 + BS - 1) / BS;
  bool bad = false;
  for (int k = threadIdx.x; k < nblk; k += NW * 32) {
    const int p = split == 0 ? ids[k] : __ldg(trow + k);   // ids[k]: this thread's own store
    bad |= (p < 0) | (p >= a.NB);
    ids[k] = p;
  }
  if (threadIdx.x < NW * NS) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
  if (threadIdx.x == 0) fence_mbar_init();
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) record_error(a.err, kDevBadBlock);
    return;
  }

  const int my_n = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;
  const uint32_t wbuf = smem_u32(smem + warp * NS * STAGE);
  const uint32_t wbar = smem_u32(&bars[warp * NS]);

  const uint64_t policy = l2_policy_evict_first();   // the KV stream is read once
  auto issue = [&](int k) {
    const int st = k % NS;
    const int p = ids[warp + NW * k];
    const int y = (p * a.Hkv + kvh) * BS;
    const uint32_t bar = wbar + 8 * st;
    const uint32_t dk = wbuf + st * STAGE;
    mbar_arrive_expect_tx(bar, STAGE);
    // one box per tile: its D/64 column boxes of BS rows land one after the
    // other (the maps' third dimension steps through them)
    tma_load_3d(dk, &tmK, 0, y, 0, bar, policy);
    tma_load_3d(dk + TILE, &tmV, 0, y, 0, bar, policy);
  };
  if (lane == 0) {
    const int pro = my_n < NS ? my_n : NS;
    for (int k = 0; k < pro; ++k) issue(k);
  }

  Compute cs;
  cs.load_q(a.q + ((size_t)seq * a.Hq + kvh * a.G) * D, a.G, lane);
  cs.reset();

  int k = 0;
  bool ok = true;
  for (; k < my_n; ++k) {
    const int st = k % NS;
    const bool done = mbar_wait(wbar + 8 * st, (k / NS) & 1);
    if (!__all_sync(kFull, done)) { ok = false; break; }
    const int jb = j0 + warp + NW * k;
    const int valid = min(BS, L - jb * BS);
    const uint32_t kt = wbuf + st * STAGE;
    if (a.k_new != nullptr && jb == (L - 1) / BS) {
      // Fused append: this step's token (position L-1) goes to its slot in
      // the cache and, since the tile was staged before, into the tile too.
      const int r = (L - 1) - jb * BS;
      const size_t src = ((size_t)seq * a.Hkv + kvh) * D;
      const size_t dst = (((size_t)ids[jb - j0] * a.Hkv + kvh) * BS + r) * D;
      for (int c = lane; c < 2 * (D / 8); c += 32) {
        const bool isv = c >= D / 8;
        const int gc = isv ? c - D / 8 : c;
        const uint4 x = *reinterpret_cast<const uint4*>((isv ? a.v_new : a.k_new) + src + gc * 8);
        const uint32_t sa = (isv ? kt + TILE : kt) + tile_off<BS>(r, gc);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sa), "r"(x.x), "r"(x.y),
                     "r"(x.z), "r"(x.w)
                     : "memory");
        *reinterpret_cast<uint4*>((isv ? a.v_cache : a.k_cache) + dst + gc * 8) = x;
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    cs.block(kt, kt + TILE, valid, a.scale_log2, lane);
    __syncwarp();
    if (lane == 0 && k + NS < my_n) {
      fence_proxy_async_smem();
      issue(k + NS);
    }
  }
  if (!ok) {
    // Give every load still in flight a bounded chance to land before the CTA
    // releases its shared memory, then report.
    const int hi = min(k + NS, my_n);
    for (int kk = k; kk < hi; ++kk) mbar_wait(wbar + 8 * (kk % NS), (kk / NS) & 1, 100000000ull);
    if (lane == 0) record_error(a.err, kDevTimeout);
  }
  // A wait that gave up fails the whole CTA: it writes no result (the merge
  // below would reuse a stage ring that a late load may still be filling).
  if (__syncthreads_or(!ok)) return;

  // Merge the warps' (m, l, o) through shared memory (the stage ring is free:
  // on this path every warp consumed every load it issued).
  float* cm = reinterpret_cast<float*>(smem);
  float* cl = cm + NW * NH;
  float* co = cl + NW * NH;
  cs.publish(cm + warp * NH, cl + warp * NH, co + warp * NH * D, lane);
  __syncthreads();

  const int nh = a.G;  // heads of this kv head's group (<= NH)
  const bool single = (L + a.P - 1) / a.P == 1;
  for (int i = threadIdx.x; i < nh * D; i += NW * 32) {
    const int h = i / D, d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[w * NH + h]);
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = fast_exp2(cm[w * NH + h] - M);
      acc = fmaf(f, co[(w * NH + h) * D + d], acc);
      lsum = fmaf(f, cl[w * NH + h], lsum);
    }
    const size_t row = (size_t)seq * a.Hq + kvh * a.G + h;
    if (single) {
      a.out[row * D + d] = to_elem<BF>(acc / lsum);
    } else {
      const size_t pr = row * a.S + split;
      a.part_o[pr * D + d] = acc;
      if (d == 0) a.part_ml[pr] = make_float2(M, lsum);
    }
  }
}

// ------------------------------------------------------------------ reduce
constexpr int kReduceThreads = 128;   // four warps: one (sequence, query head) row each

// Partials a reduce lane keeps in flight, by variant: 0 (two splits; at most
// 40 registers, so that twelve CTAs fit an idle SM) two partials; 1 (at
// most 64 registers: a CTA fits on an SM next to three decode CTAs, eight on
// an idle one) 32 floats; 2 (many splits) 64 floats.
constexpr int reduce_batch(int D, int variant) {
  return variant == 0 ? 2 : ((variant == 2 ? 64 : 32) / (D / 32) > 32 ? 32 : (variant == 2 ? 64 : 32) / (D / 32));
}
// Registers per thread the variant is built for.
constexpr int reduce_regs(int variant) { return variant == 0 ? 40 : (variant == 1 ? 64 : 128); }

// Cross-split reduce: one warp per (sequence, query head) row with more than
// one split.  M = max_s m_s, w_s = 2^(m_s - M), out = sum_s w_s o_s / sum_s
// w_s l_s, summed in split order (deterministic).  The CTAs are small, so
// that many are resident while the decode grid drains and when it completes.
// Lane j holds (m, l) of split j (of each group of 32 splits) and hands w_j
// to the other lanes by shuffle; each lane owns D / 32 output elements and
// keeps the loads of up to J partials in flight (the first batch together
// with the (m, l) loads); three builds differ only in J and their register
// budget.
template <bool BF, int D, int V>
__global__ void __launch_bounds__(kReduceThreads, 65536 / (kReduceThreads * reduce_regs(V)))
    split_reduce_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                        const int32_t* __restrict__ context_lens, uint16_t* __restrict__ out,
                        int B, int Hq, int S, int P, int max_ctx) {
  constexpr int OPL = D / 32;               // output elements per lane: 2, 4 or 8
  constexpr int J = reduce_batch(D, V);     // partials loaded per batch
  // the next kernel on the stream may become resident meanwhile
  pdl_launch_dependents();
  const int gw = blockIdx.x * (kReduceThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // The lengths were written before the decode grid started, so they can be
  // read before waiting for it; the partials only after.
  int n = 0;
  if (gw < B * Hq) {
    const int L = context_lens[gw / Hq];
    if (L >= 1 && L <= max_ctx) n = (L + P - 1) / P;
  }
  pdl_wait();
  if (n <= 1) return;
  const float2* ml = part_ml + (size_t)gw * S;
  const float* po = part_o + (size_t)gw * S * D + lane * OPL;
  // partials s_begin .. s_begin + cnt - 1 (cnt <= J) into x
  auto load = [&](float (&x)[J][OPL], int s_begin, int cnt) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      if (j < cnt) {
        const float* src = po + (size_t)(s_begin + j) * D;
#pragma unroll
        for (int e = 0; e < OPL; e += 2) {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src + e));
          x[j][e] = t.x;
          x[j][e + 1] = t.y;
        }
      }
    }
  };
  // acc += w_s x_s for the splits j0 .. of the current group of 32, w_s held by lane s % 32
  float acc[OPL];
#pragma unroll
  for (int e = 0; e < OPL; ++e) acc[e] = 0.f;
  auto accumulate = [&](const float (&x)[J][OPL], float w, int j0, int cnt) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float wj = __shfl_sync(kFull, w, (j0 + j) & 31);
      if (j0 + j < cnt) {
#pragma unroll
        for (int e = 0; e < OPL; ++e) acc[e] = fmaf(wj, x[j][e], acc[e]);
      }
    }
  };

  // The first batch of partials is in flight together with the (m, l) loads.
  float x[J][OPL];
  const int cnt0 = min(32, n);
  load(x, 0, min(J, cnt0));
  const float2 first = lane < n ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
  float M = first.x;
  for (int s = lane + 32; s < n; s += 32) M = fmaxf(M, __ldcg(ml + s).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));

  float lsum = 0.f;
  float w = lane < n ? fast_exp2(first.x - M) : 0.f;
  if (lane < n) lsum = fmaf(w, first.y, lsum);
  accumulate(x, w, 0, cnt0);
  for (int j0 = J; j0 < cnt0; j0 += J) {
    load(x, j0, min(J, cnt0 - j0));
    accumulate(x, w, j0, cnt0);
  }
  for (int s0 = 32; s0 < n; s0 += 32) {
    const bool mine = s0 + lane < n;
    const float2 v = mine ? __ldcg(ml + s0 + lane) : make_float2(0.f, 0.f);
    w = mine ? fast_exp2(v.x - M) : 0.f;
    if (mine) lsum = fmaf(w, v.y, lsum);
    const int cnt = min(32, n - s0);
    for (int j0 = 0; j0 < cnt; j0 += J) {
      load(x, s0 + j0, min(J, cnt - j0));
      accumulate(x, w, j0, cnt);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
  uint16_t* orow = out + (size_t)gw * D + lane * OPL;
#pragma unroll
  for (int e = 0; e < OPL; ++e) orow[e] = to_elem<BF>(acc[e] / lsum);
}

}  // namespace pkv
