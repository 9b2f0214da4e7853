// Launch geometry of the decode kernels, shared by the host planner and the
// kernel instantiations so that both agree on shared-memory sizes.
#pragma once

#include "pkv_internal.h"

namespace pkv {

// One pipeline stage holds a K tile and a V tile of [block_size, head_dim]
// 16-bit elements.
constexpr int stage_bytes(int D, int BS) { return 2 * BS * D * 2; }

// Warps per CTA: four for stages up to 8 KB, fewer for larger tiles, with two
// stages per warp: 64 KB of ring per CTA, so three CTAs share an SM (twelve
// warps).  Measured on GB300, this beats deeper rings with fewer warps: the
// per-SM bytes in flight are the same, the extra warps hide the per-block
// compute latency and the extra CTA covers another CTA's start-up and drain.
constexpr int geo_warps(int D, int BS) {
  return stage_bytes(D, BS) <= 8192 ? 4 : (stage_bytes(D, BS) <= 16384 ? 2 : 1);
}

// Partition kernel, per compute variant (NH = padded heads one warp
// produces: the group for the CUDA-core variant, 8 per n-tile for mma.sync).
// Tensor-core tiles of 16 or more heads (8 KB stages) need so many registers
// that only two 4-warp CTAs fit an SM; a third stage per warp restores the
// bytes in flight per SM of three 2-stage CTAs.
constexpr int part_stages(int D, int BS, int NH) {
  return (geo_warps(D, BS) == 4 && NH * D >= 2048) ? 3 : 2;
}
// Stage ring + one mbarrier per stage + the partition's block ids + 1 KB of
// slack for aligning the ring to the 1024-byte swizzle atom, grown when the
// warps' (m, l, o) merge needs more room than the ring.
constexpr int part_smem(int D, int BS, int NH) {
  return geo_warps(D, BS) * part_stages(D, BS, NH) * stage_bytes(D, BS) +
         geo_warps(D, BS) * part_stages(D, BS, NH) * 8 + kMaxBlocksPerCta * 4 + 1024 +
         (geo_warps(D, BS) * NH * (D + 2) * 4 >
                  geo_warps(D, BS) * part_stages(D, BS, NH) * stage_bytes(D, BS)
              ? ((geo_warps(D, BS) * NH * (D + 2) * 4 -
                  geo_warps(D, BS) * part_stages(D, BS, NH) * stage_bytes(D, BS) + 15) &
                 ~15)
              : 0);
}
// Padded heads per warp of a variant (0 CUDA cores, 1 mma.sync) for group G.
constexpr int compute_heads(int variant, int G) {
  return variant == 0 ? G : 8 * (G <= 8 ? 1 : (G <= 16 ? 2 : 4));
}

// Resident CTAs per SM for a dynamic shared-memory size (228 KB per SM, 1 KB
// reserved per CTA, at most 16 CTAs of these sizes).
constexpr int ctas_per_sm_for(int smem) {
  return (233472 / (smem + 1024)) < 16 ? 233472 / (smem + 1024) : 16;
}

}  // namespace pkv
