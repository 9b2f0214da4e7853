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

constexpr int geo_stages(int /*D*/, int /*BS*/) { return 2; }

// Stage ring + one mbarrier per stage + the partition's block ids + 1 KB of
// slack for aligning the ring to the 1024-byte swizzle atom.
constexpr int geo_smem(int D, int BS) {
  return geo_warps(D, BS) * geo_stages(D, BS) * stage_bytes(D, BS) +
         geo_warps(D, BS) * geo_stages(D, BS) * 8 + kMaxBlocksPerCta * 4 + 1024;
}

// Largest batch the persistent schedule takes (its per-sequence block prefix
// lives in shared memory); larger batches use the fixed-partition schedule.
constexpr int kPersistMaxSeqs = 2048;

// Persistent kernel: stage ring + mbarriers + per-stage (unit, block) tags +
// the block prefix cum[0..B] + alignment slack.
constexpr int geo_persist_smem(int D, int BS, int B) {
  return geo_warps(D, BS) * geo_stages(D, BS) * stage_bytes(D, BS) +
         geo_warps(D, BS) * geo_stages(D, BS) * 16 + (B + 1) * 4 + 1024;
}

// Resident CTAs per SM for a dynamic shared-memory size (228 KB per SM, 1 KB
// reserved per CTA, at most 16 CTAs of these sizes).
constexpr int ctas_per_sm_for(int smem) {
  return (233472 / (smem + 1024)) < 16 ? 233472 / (smem + 1024) : 16;
}

}  // namespace pkv
