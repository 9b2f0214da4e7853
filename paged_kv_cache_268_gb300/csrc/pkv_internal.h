// Internal interface between the C-ABI front end (pkv_api.cu) and the decode
// kernel translation units (pkv_decode_inst.cu, compiled once per element
// type and kernel variant).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Device error word codes (mirror PKV_DEV_* in include/pkv.h).
enum : int { kDevBadBlock = 1, kDevBadContext = 2, kDevBadSlot = 3, kDevTimeout = 4 };

// Largest number of KV blocks one CTA's partition may span.
constexpr int kMaxBlocksPerCta = 256;

struct DecodeArgs {
  const uint16_t* q;            // [B, Hq, D]
  const int32_t* block_tables;  // [B, MB]
  const int32_t* context_lens;  // [B]
  uint16_t* out;                // [B, Hq, D]
  float* part_o;                // un-normalised partial outputs [B, Hq, S, D]
  float2* part_ml;              // (running max in log2 units, sum) per partial row
  const uint16_t* k_new;        // fused append: this step's K/V rows [B, Hkv, D],
  const uint16_t* v_new;        //   or null for a plain decode
  uint16_t* k_cache;            // fused append: the caches the rows go to
  uint16_t* v_cache;
  int* err;                     // device error word
  int B, Hq, Hkv, G, MB, NB;
  int S;                        // splits per sequence (grid extent)
  int P;                        // tokens per split, multiple of the block size
  int max_ctx;                  // upper bound on every context length
  float scale_log2;             // softmax scale * log2(e)
};

// Per-(head_dim, block_size, variant) launch geometry.
struct KernelGeometry {
  int warps;        // warps per CTA, each with its own KV pipeline
  int stages;       // pipeline stages per warp (one K tile + one V tile each)
  int smem_bytes;   // dynamic shared memory per CTA
};

// Variant: 0 = CUDA-core kernel (group size 1 or 2), 1 = mma.sync tensor-core
// kernel (group size 1..32), 2 = tcgen05 kernel (its geometry is its own).
bool decode_geometry(int head_dim, int block_size, int variant, int group_size,
                     KernelGeometry* g);

// Launch the decode kernel over the grid B * Hkv * S of (sequence, kv head,
// partition) units.  Returns cudaErrorInvalidValue for an unbuilt combination.
cudaError_t launch_decode_f16_simt(const DecodeArgs&, const CUtensorMap&, const CUtensorMap&,
                                   int head_dim, int block_size, cudaStream_t);
cudaError_t launch_decode_bf16_simt(const DecodeArgs&, const CUtensorMap&, const CUtensorMap&,
                                    int head_dim, int block_size, cudaStream_t);
cudaError_t launch_decode_f16_mma(const DecodeArgs&, const CUtensorMap&, const CUtensorMap&,
                                  int head_dim, int block_size, cudaStream_t);
cudaError_t launch_decode_bf16_mma(const DecodeArgs&, const CUtensorMap&, const CUtensorMap&,
                                   int head_dim, int block_size, cudaStream_t);

// tcgen05 variant (head_dim 128, group size up to 32): same grid and
// partitions as the other variants; it walks a partition in 128-token groups
// (the last one may be ragged).
cudaError_t launch_decode_tc(const DecodeArgs&, const CUtensorMap&, const CUtensorMap&, bool bf16,
                             int head_dim, int block_size, cudaStream_t);
int tc_smem_bytes(int group_size);
int tc_ring_slots(int group_size);   // 32 KB K/V tile slots per CTA
int tc_warps(int group_size);        // warps per CTA (softmax, producer, MMA)

int* device_error_word();  // device address of the error word (current device)

}  // namespace pkv
