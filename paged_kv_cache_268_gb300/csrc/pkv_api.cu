// C-ABI front end of libpkv: argument validation, split-KV planning, TMA
// descriptor encoding, and the KV append and cross-split reduce launches.
// The declarations and the contract of every entry point are in include/pkv.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "pkv_decode.cuh"
#include "pkv_geometry.h"
#include "pkv_internal.h"

namespace pkv {

__device__ int g_device_error;

namespace {

std::atomic<uint64_t> g_launches{0};

// ------------------------------------------------------------------ append
// KV append scatter (block manager slot write): one warp per (token, kv head)
// row; the warp copies the K row then the V row with 16-byte vector stores.
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     const int32_t* __restrict__ slot_mapping, uint4* __restrict__ k_cache,
                     uint4* __restrict__ v_cache, int T, int Hkv, int bs, int NB,
                     int chunks_per_row, int* err) {
  // a decode launched next on the stream may become resident meanwhile; it
  // waits for this grid before reading the cache
  pdl_launch_dependents();
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(T) * Hkv) return;
  const int t = static_cast<int>(row / Hkv);
  const int h = static_cast<int>(row - static_cast<long long>(t) * Hkv);
  const int s = slot_mapping[t];
  if (s < 0) return;
  if (static_cast<long long>(s) >= static_cast<long long>(NB) * bs) {
    if (lane == 0 && h == 0) record_error(err, kDevBadSlot);
    return;
  }
  const size_t dst = ((static_cast<size_t>(s / bs) * Hkv + h) * bs + (s % bs)) * chunks_per_row;
  const size_t src = static_cast<size_t>(row) * chunks_per_row;
  for (int c = lane; c < 2 * chunks_per_row; c += 32) {
    if (c < chunks_per_row) {
      k_cache[dst + c] = k[src + c];
    } else {
      const int cc = c - chunks_per_row;
      v_cache[dst + cc] = v[src + cc];
    }
  }
}

// ------------------------------------------------------------------ self-test
// One warp waits on an mbarrier that nothing arrives on, with the same
// bounded wait as the decode kernels, and reports the timeout.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait(smem_u32(&bar), 0, limit_ns);
  if (!__all_sync(kFull, done) && threadIdx.x == 0) record_error(err, kDevTimeout);
}

// ------------------------------------------------------------------ block copy
// Whole-block copy between pools (copy-on-write within the GPU pool, swap-out
// to and swap-in from a pinned CPU pool that the GPU reaches directly): pair
// i copies block pairs[2i] of the source pool to block pairs[2i+1] of the
// destination pool, every kv head, K and V.  CTA (i, K|V, part) moves up to
// 16 KB with four independent 16-byte loads per thread before the stores.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                       uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                       const int32_t* __restrict__ pairs, int src_nb, int dst_nb,
                       int chunks_per_block, int* err) {
  const int pair = blockIdx.x >> 1;
  const bool is_v = blockIdx.x & 1;
  const int s = pairs[2 * pair], d = pairs[2 * pair + 1];
  if (s < 0 || s >= src_nb || d < 0 || d >= dst_nb) {
    if (threadIdx.x == 0 && !is_v && blockIdx.y == 0) record_error(err, kDevBadBlock);
    return;
  }
  const uint4* src = (is_v ? src_v : src_k) + (size_t)s * chunks_per_block;
  uint4* dst = (is_v ? dst_v : dst_k) + (size_t)d * chunks_per_block;
  const int base = blockIdx.y * 1024 + threadIdx.x;
  uint4 x[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = base + u * 256;
    if (c < chunks_per_block) x[u] = src[c];
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = base + u * 256;
    if (c < chunks_per_block) dst[c] = x[u];
  }
}

// ------------------------------------------------------------------ reduce
// Launch a dependent kernel with programmatic stream serialisation: it may
// start launching while the decode kernel's last CTAs still run, and waits
// (griddepcontrol.wait) for that grid before reading its partials.
template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, cudaStream_t stream,
                             Args... args) {
  static_assert(sizeof...(KArgs) == sizeof...(Args), "argument count");
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Reduce grid: one warp per (sequence, query head) row.  The smallest
// variant that loads every partial of a row in one batch: two splits (the
// 40-register build, so that the most warps are resident), up to the 64-
// register build's batch, else the 128-register build.
template <bool BF, int D>
cudaError_t launch_reduce_d(const DecodeArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.Hq;
  const int warps = kReduceThreads / 32;
  const unsigned g = static_cast<unsigned>((rows + warps - 1) / warps);
  auto kern = a.S <= reduce_batch(D, 1) ? split_reduce_kernel<BF, D, 1>
                                         : split_reduce_kernel<BF, D, 2>;
  if constexpr (D <= 128) {   // at head_dim 256 the 40-register build would spill
    if (a.S <= reduce_batch(D, 0)) kern = split_reduce_kernel<BF, D, 0>;
  }
  return launch_dependent(kern, g, stream, a.part_o, a.part_ml, a.context_lens, a.out, a.B, a.Hq,
                          a.S, a.P, a.max_ctx);
}

template <bool BF>
cudaError_t launch_reduce(const DecodeArgs& a, int D, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_reduce_d<BF, 64>(a, stream);
    case 128: return launch_reduce_d<BF, 128>(a, stream);
    case 256: return launch_reduce_d<BF, 256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------------ devices
struct DeviceInfo {
  bool valid = false;
  int sms = 0;
  int* err = nullptr;
  // workspace set with pkv_set_workspace (caller-owned; null when none)
  void* ws = nullptr;
  size_t ws_bytes = 0;
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

int current_device(DeviceInfo** info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return PKV_ERR_CUDA;
    d.err = static_cast<int*>(p);
    d.valid = true;
  }
  *info = &d;
  return PKV_OK;
}

// ------------------------------------------------------------------ TMA maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? PKV_OK : PKV_ERR_CUDA;
}

// The pool [NB, Hkv, bs, D] as a 2-D tensor of NB * Hkv * bs rows of D
// elements; one box is 64 elements (128 bytes) x bs rows with the 128-byte
// swizzle, so one [bs, D] tile is D / 64 boxes.
// The cache [NB * Hkv * bs rows][D] seen as 64-element column boxes of bs
// rows, 128-byte swizzled.  Two forms: 2-D (x = column, y = row; one box per
// load, for the tcgen05 kernel, whose tiles keep the column boxes of 128
// tokens apart) and 3-D (x = column within a box, y = row, z = box: a load
// of one block's tile brings its D / 64 column boxes one after the other, as
// the partition kernel stages them).
int encode_cache_map(CUtensorMap* map, const void* base, const pkv_shape& s, bool three_d) {
  const cuuint64_t rows = static_cast<cuuint64_t>(s.num_blocks) * s.num_kv_heads * s.block_size;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(s.head_dim) * 2;
  const CUtensorMapDataType dt =
      s.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (three_d) {
    cuuint64_t dims[3] = {64, rows, static_cast<cuuint64_t>(s.head_dim / 64)};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(s.block_size),
                         static_cast<cuuint32_t>(s.head_dim / 64)};
    r = g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.head_dim), rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(s.block_size)};
    r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

struct MapCacheEntry {
  const void* base = nullptr;
  pkv_shape shape{};
  int device = -1;
  bool three_d = false;
  CUtensorMap map{};
};
std::mutex g_map_mutex;
MapCacheEntry g_map_cache[8];
int g_map_next = 0;

int cache_map(CUtensorMap* out, const void* base, const pkv_shape& s, bool three_d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  for (auto& e : g_map_cache) {
    if (e.base == base && e.device == dev && e.three_d == three_d &&
        e.shape.num_blocks == s.num_blocks &&
        e.shape.num_kv_heads == s.num_kv_heads && e.shape.block_size == s.block_size &&
        e.shape.head_dim == s.head_dim && e.shape.dtype == s.dtype) {
      *out = e.map;
      return PKV_OK;
    }
  }
  MapCacheEntry& e = g_map_cache[g_map_next];
  g_map_next = (g_map_next + 1) % 8;
  int rc = encode_cache_map(&e.map, base, s, three_d);
  if (rc != PKV_OK) {
    e.base = nullptr;
    return rc;
  }
  e.base = base;
  e.shape = s;
  e.device = dev;
  e.three_d = three_d;
  *out = e.map;
  return PKV_OK;
}

// ------------------------------------------------------------------ checks
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache_shape(const pkv_shape* s) {
  if (!s) return PKV_ERR_NULL;
  if (s->num_kv_heads < 1 || s->head_dim < 1 || s->block_size < 1 || s->num_blocks < 1)
    return PKV_ERR_INVALID;
  if (s->dtype != PKV_F16 && s->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (s->head_dim != 64 && s->head_dim != 128 && s->head_dim != 256) return PKV_ERR_UNSUPPORTED;
  if (s->block_size != 16 && s->block_size != 32) return PKV_ERR_UNSUPPORTED;
  // TMA row coordinates are 32-bit signed
  if (static_cast<long long>(s->num_blocks) * s->num_kv_heads * s->block_size >= (1ll << 31))
    return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

int check_decode_shape(const pkv_shape* s) {
  int rc = check_cache_shape(s);
  if (rc != PKV_OK) return rc;
  if (s->num_seqs < 0 || s->num_q_heads < 1 || s->max_blocks_per_seq < 1 ||
      s->max_context_len < 1 || s->split_tokens < 0 || s->kernel < 0 || s->kernel > 3)
    return PKV_ERR_INVALID;
  if (s->num_q_heads % s->num_kv_heads != 0) return PKV_ERR_INVALID;
  if (static_cast<long long>(s->max_context_len) >
      static_cast<long long>(s->max_blocks_per_seq) * s->block_size)
    return PKV_ERR_INVALID;
  const int G = s->num_q_heads / s->num_kv_heads;
  if (G > 32) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

// Inner-loop variant (0 CUDA cores, 1 mma.sync, 2 tcgen05) for a shape, or -1
// when the requested one cannot run it.  Every variant serves the plain
// decode and the fused step.
int pick_variant(const pkv_shape* s) {
  const int G = s->num_q_heads / s->num_kv_heads;
  const bool tc_ok = s->head_dim == 128 && G <= 32;
  switch (s->kernel) {
    case 1: return G <= 2 ? 0 : -1;
    case 2: return 1;
    case 3: return tc_ok ? 2 : -1;
    default:
      // Measured on GB300 (whole step, steps back to back): mma.sync stays ahead of the
      // tcgen05 kernel at every group size (Llama-3-8B-shaped batch, group 4:
      // 114.7 vs 188.4 us; long context, group 8: 82.5 vs 84.2 us; 128/8
      // heads: 104.1 vs 120.7 us; 256/8 heads: 143.3 vs 174.1 us), so the
      // library's choice never takes tcgen05.
      return G <= 2 ? 0 : 1;
  }
}

int make_plan(const pkv_shape* s, int sms, pkv_plan* plan) {
  const int G = s->num_q_heads / s->num_kv_heads;
  const int bs = s->block_size;
  plan->variant = pick_variant(s);
  if (plan->variant < 0) return PKV_ERR_UNSUPPORTED;
  KernelGeometry geo{};
  decode_geometry(s->head_dim, bs, plan->variant, G, &geo);
  if (plan->variant == 2) {
    geo.warps = tc_warps(G);
    geo.stages = tc_ring_slots(G);   // K/V tile slots of 128 tokens
    geo.smem_bytes = tc_smem_bytes(G);
  }
  plan->warps_per_cta = geo.warps;
  plan->stages_per_warp = geo.stages;
  const long long units = static_cast<long long>(s->num_seqs) * s->num_kv_heads;
  plan->schedule = 0;
  const int maxL = s->max_context_len;
  // every warp gets the same block count; the tcgen05 kernel walks 128-token groups
  const int gran = plan->variant == 2 ? 128 : bs * geo.warps;
  const int cap = kMaxBlocksPerCta * bs;      // ids of one partition fit in shared memory
  long long P;
  if (s->split_tokens > 0) {
    P = (static_cast<long long>(s->split_tokens) + bs - 1) / bs * bs;
  } else {
    // 1024-token partitions keep every CTA long enough to amortise its
    // start-up while the hardware block scheduler balances the SMs.  When
    // the whole grid would be under four waves, wave quantisation dominates
    // instead: use exactly one wave of equal partitions.
    const long long slots = static_cast<long long>(sms) * ctas_per_sm_for(geo.smem_bytes);
    // the tcgen05 kernel's CTAs start up slower (TMEM, a deeper ring, fewer
    // CTAs per SM): 2048-token partitions, 4096 where one CTA fills an SM.
    // The 16- and 32-head mma.sync tiles (two CTAs per SM) also run best on
    // 2048 (measured on one GB300: 5% faster than 1024 at 32 heads, 2% at 16;
    // 3072 and 4096 slower again).
    const bool wide_mma = plan->variant == 1 && G > 8;
    if (plan->variant == 2)
      P = G > 16 ? 4096 : 2048;
    else
      P = wide_mma ? 2048 : 1024;
    // one wave when the grid would be under four waves (two for the wide
    // mma.sync tiles, which measured faster at 3.4 waves than at one).  The
    // two-warp CTAs of 16 KB stages fill that wave at two CTAs per SM, the
    // others at every CTA an SM holds: measured on one GB300, the 4 x 32768
    // long-context batch ran 1.2% faster at two (288 CTAs) than at three (448),
    // a 2-sequence cut of it 4% faster, while the four-warp CTAs of 8 KB stages
    // ran 15-18% slower at two.
    const long long min_waves = wide_mma ? 2 : 4;
    if (units > 0 && units * ((maxL + P - 1) / P) < min_waves * slots) {
      const long long wave =
          plan->variant != 2 && geo.warps == 2 && ctas_per_sm_for(geo.smem_bytes) > 2 ? 2LL * sms
                                                                                   : slots;
      const long long S = wave / units > 0 ? wave / units : 1;
      P = (maxL + S - 1) / S;
    }
    P = (P + gran - 1) / gran * gran;
    // At most 1024 partitions per sequence.
    const long long pmin = (static_cast<long long>(maxL) + 1023) / 1024;
    if (P < pmin) P = (pmin + gran - 1) / gran * gran;
  }
  if (P > cap) P = cap;
  if (P > maxL) P = (maxL + bs - 1) / bs * bs;
  if (P < bs) P = bs;
  plan->split_tokens = static_cast<int32_t>(P);
  plan->num_splits = static_cast<int32_t>((maxL + P - 1) / P);
  const long long grid = units * plan->num_splits;
  if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  // output rows (sequence, query head) are indexed in 32 bits by the reduce
  if (static_cast<long long>(s->num_seqs) * s->num_q_heads > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  plan->grid_ctas = static_cast<int32_t>(grid);
  plan->workspace_bytes =
      plan->num_splits > 1
          ? static_cast<size_t>(s->num_seqs) * s->num_q_heads * plan->num_splits *
                (static_cast<size_t>(s->head_dim) * 4 + 8)
          : 0;
  return PKV_OK;
}

}  // namespace

bool decode_geometry(int D, int BS, int variant, int G, KernelGeometry* g) {
  const int nh = compute_heads(variant, G);
  g->warps = geo_warps(D, BS);
  g->stages = part_stages(D, BS, nh);
  g->smem_bytes = part_smem(D, BS, nh);
  return true;
}

// The workspace set for the current device, or {nullptr, 0}.
static void set_workspace_of(DeviceInfo* d, void** ptr, size_t* bytes) {
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  *ptr = d->ws;
  *bytes = d->ws_bytes;
}

int* device_error_word() {
  DeviceInfo* d = nullptr;
  return current_device(&d) == PKV_OK ? d->err : nullptr;
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_version(void) { return 100; }

extern "C" uint64_t pkv_launch_count(void) { return g_launches.load(); }

extern "C" const char* pkv_strerror(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_INVALID: return "invalid size (non-positive dimension, Hq % Hkv != 0, or max_context_len > max_blocks_per_seq * block_size)";
    case PKV_ERR_UNSUPPORTED: return "unsupported head_dim, block_size, group size, dtype or pool size";
    case PKV_ERR_ALIGN: return "a pointer is not 16-byte (arrays of 16-bit elements) or 4-byte (int32 arrays) aligned";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than pkv_workspace_bytes";
    case PKV_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case PKV_ERR_DEVICE: return "a kernel recorded a device-side error";
    case PKV_ERR_NO_BLOCKS: return "the block pool has no free block left";
    default: return "unknown pkv error code";
  }
}

extern "C" int pkv_decode_plan(const pkv_shape* s, pkv_plan* plan) {
  if (!s || !plan) return PKV_ERR_NULL;
  int rc = check_decode_shape(s);
  if (rc != PKV_OK) return rc;
  DeviceInfo* d = nullptr;
  rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  return make_plan(s, d->sms, plan);
}

extern "C" int pkv_decode_plan_for(const pkv_shape* s, int32_t num_sms, pkv_plan* plan) {
  if (!s || !plan) return PKV_ERR_NULL;
  if (num_sms < 1) return PKV_ERR_INVALID;
  const int rc = check_decode_shape(s);
  if (rc != PKV_OK) return rc;
  return make_plan(s, num_sms, plan);
}

extern "C" int pkv_workspace_bytes(const pkv_shape* s, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  pkv_plan plan{};
  int rc = pkv_decode_plan(s, &plan);
  if (rc != PKV_OK) return rc;
  *bytes = plan.workspace_bytes;
  return PKV_OK;
}

extern "C" int pkv_set_workspace(void* dev_ptr, size_t bytes) {
  if (dev_ptr != nullptr) {
    if (bytes == 0) return PKV_ERR_INVALID;
    if (!aligned(dev_ptr, 16)) return PKV_ERR_ALIGN;
  }
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  if (dev_ptr != nullptr) {
    // it must be memory of the current device (not host memory, not another GPU's)
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, dev_ptr) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_INVALID;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev)
      return PKV_ERR_INVALID;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  d->ws = dev_ptr;
  d->ws_bytes = dev_ptr ? bytes : 0;
  return PKV_OK;
}

extern "C" int pkv_kv_cache_append(const pkv_shape* s, const void* k, const void* v,
                                   const int32_t* slot_mapping, int32_t num_tokens,
                                   void* k_cache, void* v_cache, pkv_stream_t stream) {
  int rc = check_cache_shape(s);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return PKV_ERR_INVALID;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 4))
    return PKV_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  const long long rows = static_cast<long long>(num_tokens) * s->num_kv_heads;
  const long long grid = (rows + 7) / 8;
  if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  kv_append_kernel<<<static_cast<unsigned>(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_tokens, s->num_kv_heads,
      s->block_size, s->num_blocks, s->head_dim / 8, d->err);
  g_launches.fetch_add(1);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

namespace {

// Shared body of pkv_paged_attn_decode and pkv_decode_step (k_new != null).
int decode_impl(const pkv_shape* s, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, float scale, void* out,
                void* workspace, size_t workspace_bytes, pkv_stream_t stream, const void* k_new,
                const void* v_new) {
  int rc = check_decode_shape(s);
  if (rc != PKV_OK) return rc;
  if (s->num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_ERR_NULL;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_ERR_ALIGN;
  DeviceInfo* d = nullptr;
  rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  pkv_plan plan{};
  rc = make_plan(s, d->sms, &plan);
  if (rc != PKV_OK) return rc;
  if (plan.workspace_bytes > 0) {
    if (!workspace) set_workspace_of(d, &workspace, &workspace_bytes);
    if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 16))
      return PKV_ERR_WORKSPACE;
  }
  rc = get_encoder();
  if (rc != PKV_OK) return rc;
  CUtensorMap tk, tv;
  const bool three_d = plan.variant != 2;
  rc = cache_map(&tk, k_cache, *s, three_d);
  if (rc != PKV_OK) return rc;
  rc = cache_map(&tv, v_cache, *s, three_d);
  if (rc != PKV_OK) return rc;

  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = static_cast<uint16_t*>(out);
  const int G = s->num_q_heads / s->num_kv_heads;
  {
    const size_t rows = static_cast<size_t>(s->num_seqs) * s->num_q_heads * plan.num_splits;
    a.part_o = plan.workspace_bytes ? static_cast<float*>(workspace) : nullptr;
    a.part_ml = plan.workspace_bytes ? reinterpret_cast<float2*>(static_cast<float*>(workspace) +
                                                                 rows * s->head_dim)
                                     : nullptr;
  }
  a.err = d->err;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_cache = static_cast<uint16_t*>(const_cast<void*>(k_cache));
  a.v_cache = static_cast<uint16_t*>(const_cast<void*>(v_cache));
  a.B = s->num_seqs;
  a.Hq = s->num_q_heads;
  a.Hkv = s->num_kv_heads;
  a.G = G;
  a.MB = s->max_blocks_per_seq;
  a.NB = s->num_blocks;
  a.S = plan.num_splits;
  a.P = plan.split_tokens;
  a.max_ctx = s->max_context_len;
  a.scale_log2 = scale * 1.4426950408889634f;  // log2(e)

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = s->dtype == PKV_BF16;
  const int D = s->head_dim, BS = s->block_size;
  cudaError_t e;
  if (plan.variant == 2)
    e = launch_decode_tc(a, tk, tv, bf, D, BS, st);
  else if (plan.variant == 0)
    e = bf ? launch_decode_bf16_simt(a, tk, tv, D, BS, st)
           : launch_decode_f16_simt(a, tk, tv, D, BS, st);
  else
    e = bf ? launch_decode_bf16_mma(a, tk, tv, D, BS, st)
           : launch_decode_f16_mma(a, tk, tv, D, BS, st);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  g_launches.fetch_add(1);
  if (plan.num_splits > 1) {
    e = bf ? launch_reduce<true>(a, D, st) : launch_reduce<false>(a, D, st);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attn_decode(const pkv_shape* s, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, float scale, void* out,
                                     void* workspace, size_t workspace_bytes,
                                     pkv_stream_t stream) {
  return decode_impl(s, q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                     workspace_bytes, stream, nullptr, nullptr);
}

extern "C" int pkv_decode_step(const pkv_shape* s, const void* q, const void* k_new,
                               const void* v_new, void* k_cache, void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               pkv_stream_t stream) {
  if (!s) return PKV_ERR_NULL;
  if (s->num_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_NULL;
  if (s->num_seqs > 0 && (!aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_ALIGN;
  return decode_impl(s, q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                     workspace_bytes, stream, k_new, v_new);
}

extern "C" int pkv_copy_blocks(const pkv_shape* s, const void* src_k, const void* src_v,
                               int32_t src_num_blocks, void* dst_k, void* dst_v,
                               int32_t dst_num_blocks, const int32_t* pairs, int32_t num_pairs,
                               pkv_stream_t stream) {
  if (!s) return PKV_ERR_NULL;
  if (s->num_kv_heads < 1 || s->head_dim < 1 || s->block_size < 1 || src_num_blocks < 1 ||
      dst_num_blocks < 1 || num_pairs < 0)
    return PKV_ERR_INVALID;
  if (s->dtype != PKV_F16 && s->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (s->head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PKV_OK;
  if (!src_k || !src_v || !dst_k || !dst_v || !pairs) return PKV_ERR_NULL;
  if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16) ||
      !aligned(pairs, 4))
    return PKV_ERR_ALIGN;
  const long long chunks = static_cast<long long>(s->num_kv_heads) * s->block_size * s->head_dim / 8;
  if (chunks > (1ll << 30) || num_pairs > (1 << 30)) return PKV_ERR_UNSUPPORTED;
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  const dim3 grid(2u * static_cast<unsigned>(num_pairs), static_cast<unsigned>((chunks + 1023) / 1024));
  copy_blocks_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
      static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), pairs, src_num_blocks,
      dst_num_blocks, static_cast<int>(chunks), d->err);
  g_launches.fetch_add(1);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_selftest_wait_timeout(int32_t limit_us, pkv_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return PKV_ERR_INVALID;
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      d->err, static_cast<unsigned long long>(limit_us) * 1000ull);
  g_launches.fetch_add(1);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_get_device_error(int32_t* code, pkv_stream_t stream) {
  if (!code) return PKV_ERR_NULL;
  DeviceInfo* d = nullptr;
  int rc = current_device(&d);
  if (rc != PKV_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, d->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaMemsetAsync(d->err, 0, sizeof(int), st) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
  *code = host;
  return PKV_OK;
}
