// pkv_paged_attn_decode_noalloc: paged decode attention for callers that
// cannot allocate device memory.
//
// The regular entry point asks the caller for a workspace (the split-KV
// partials).  Some callers have no way to provide one: a serving engine that
// reserved all of HBM for its KV block pool at start-up and hands its kernel
// libraries no allocator, or code on a latency-critical path where cudaMalloc
// (which can synchronise the whole device) is not acceptable.  This entry point
// needs nothing from them but inputs and outputs: the partials live in a
// fixed-size array in the library's own device memory, reserved once when the
// library is loaded on a GPU and held until the process exits.
//
// Properties a caller has to know:
//  - Limit: the partials of one call must fit in kNoAllocScratchBytes (64 MiB);
//    larger calls are rejected with PKV_ERR_WORKSPACE before anything is
//    enqueued.  A larger split_tokens shrinks the partials.
//  - Set-up: the first call on each device looks up the array's device
//    address (cudaGetSymbolAddress) with that device current, and remembers
//    it.  Make that first call before any stream capture.
//  - Sharing: every call on a device uses the same array, and it keeps the
//    previous call's contents.  Nothing in it has to start at zero (each
//    partial is written by the decode kernel before the reduce kernel reads it
//    within the same call), but two calls whose work overlaps on the GPU (on
//    different streams, or from different host threads) race on it.
//  - It never calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "pkv.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device (set up once per
// device), or nullptr if the lookup failed.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" int pkv_paged_attn_decode_noalloc(const pkv_shape* shape, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             void* out, pkv_stream_t stream) {
  pkv_plan plan{};
  int rc = pkv_decode_plan(shape, &plan);
  if (rc != PKV_OK) return rc;
  if (plan.workspace_bytes > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (plan.workspace_bytes > 0) {
    scratch = noalloc_scratch();
    if (!scratch) return PKV_ERR_CUDA;
  }
  return pkv_paged_attn_decode(shape, q, k_cache, v_cache, block_tables, context_lens, scale,
                               out, scratch, kNoAllocScratchBytes, stream);
}
