/*
 * pkv — paged KV-cache decode attention for GB300 (sm_103a), C ABI.
 *
 * The problem these calls solve is stated in the "PagedAttention" section of
 * the third page (bbs.pinggu.org thread 16345627, "memory management as an
 * operating system"): the KV cache of every sequence is cut into fixed-size
 * physical blocks that need not be contiguous in device memory, a per-sequence
 * block table maps logical blocks to physical ones, and the attention kernel
 * reaches K/V by looking the block up in the table (indirect addressing).  The
 * attention itself is softmax(q . K^T * scale) . V (second page, "model
 * executor" article, section 3.1); a decode step has one query token per
 * sequence, so there is no mask.  New tokens enter the cache through the block
 * manager's slots (first page, section 4.2) once per scheduler iteration
 * (third page, "continuous batching").
 *
 * Conventions for every call
 *  - All array arguments are DEVICE pointers owned by the caller; the library
 *    never frees or retains them.  Layouts are dense and row-major.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  No call synchronises the host, except pkv_get_device_error.
 *  - Calls return PKV_OK (0) or a negative PKV_ERR_* code.  Argument errors are
 *    detected on the host before anything is enqueued.  The CONTENTS of device
 *    arrays (block ids, slots, lengths) cannot be checked on the host without a
 *    sync; the kernels check them instead, skip the offending unit and record
 *    a code in a device-side error word read by pkv_get_device_error.
 *  - Both calls are deterministic: the same inputs give bit-identical outputs.
 *  - Calls enqueued on one stream run in order, so a decode enqueued after an
 *    append on the same stream sees the appended tokens.
 *
 * Element type: q, k, v, k_cache, v_cache and out all share one 16-bit type,
 * IEEE binary16 (PKV_F16) or bfloat16 (PKV_BF16).  Arithmetic is FP32 with
 * round-to-nearest-even on the final store.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared here so that callers need no CUDA
 * header. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

enum {
  PKV_OK = 0,
  PKV_ERR_NULL = -1,         /* a required pointer is NULL */
  PKV_ERR_INVALID = -2,      /* a size is out of range, or Hq % Hkv != 0 */
  PKV_ERR_UNSUPPORTED = -3,  /* head_dim, block_size, group size or dtype not built */
  PKV_ERR_ALIGN = -4,        /* a pointer is not aligned as the layout requires */
  PKV_ERR_WORKSPACE = -5,    /* workspace missing or smaller than required */
  PKV_ERR_CUDA = -6,         /* a CUDA runtime/driver call failed */
  PKV_ERR_DEVICE = -7,       /* reserved: a kernel recorded a device-side error */
  PKV_ERR_NO_BLOCKS = -8     /* block manager: the pool has no free block left */
};

/* Device-side error codes (pkv_get_device_error). */
enum {
  PKV_DEV_OK = 0,
  PKV_DEV_BAD_BLOCK_ID = 1,  /* a block table entry outside [0, num_blocks) */
  PKV_DEV_BAD_CONTEXT = 2,   /* a context length outside [1, max_context_len] */
  PKV_DEV_BAD_SLOT = 3,      /* a slot >= num_blocks * block_size */
  PKV_DEV_TIMEOUT = 4        /* a pipeline wait gave up (should never happen) */
};

/* Shape of one paged cache and of the batch that reads it.
 *   num_seqs            B, sequences in the batch (one query token each)
 *   num_q_heads         Hq
 *   num_kv_heads        Hkv; Hq % Hkv == 0; query head h reads kv head
 *                       h / (Hq / Hkv) (contiguous grouping); the group
 *                       size Hq / Hkv is at most 32
 *   head_dim            D, one of 64, 128, 256
 *   block_size          bs, tokens per physical block, one of 16, 32
 *   num_blocks          NB, physical blocks in the pool
 *   max_blocks_per_seq  MB, row stride of block_tables
 *   max_context_len     host-known upper bound on every context_lens[i]
 *                       (1 <= it <= MB * bs); sizes the split-KV grid
 *   dtype               pkv_dtype
 *   split_tokens        split-KV partition size: 0 lets the library choose;
 *                       > 0 sets the tokens per partition (rounded up to a
 *                       multiple of bs; the tcgen05 kernel walks a partition
 *                       in 128-token groups, the last of which may be
 *                       ragged).  Negative values give PKV_ERR_INVALID.
 *   kernel              inner-loop choice: 0 lets the library choose, 1 CUDA
 *                       cores (group size 1-2), 2 mma.sync tensor cores
 *                       (group 3-32), 3 tcgen05 tensor cores with TMEM
 *                       accumulators (head_dim 128, group 1-32; decode or
 *                       fused step).  The library's choice: 1 for groups
 *                       of 1-2, 2 for 3-32 (faster than 3 on GB300 at every
 *                       group size measured).  An inapplicable choice gives
 *                       PKV_ERR_UNSUPPORTED. */
typedef struct {
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_context_len;
  int32_t dtype;
  int32_t split_tokens;
  int32_t kernel;
} pkv_shape;

/* How a decode call will run (filled by pkv_decode_plan).  One CTA per
 * (sequence, kv head, partition of split_tokens tokens), grid_ctas =
 * B * Hkv * S, dispatched by the hardware as SMs free up, then a
 * cross-partition reduce kernel when S > 1.  With split_tokens == 0 the
 * partition is 1024 tokens (2048 for the 16- and 32-head mma.sync tiles,
 * 2048/4096 for the tcgen05 kernel with 16/32 padded heads), or one wave of
 * equal partitions when the grid would be under four waves (two for the wide
 * mma.sync tiles); a wave is every CTA the SMs hold, or two per SM for the
 * two-warp CTAs of 16 KB stages (head_dim 128 with block size 32, head_dim
 * 256 with block size 16). */
typedef struct {
  int32_t schedule;         /* always 0 (the partition schedule) */
  int32_t split_tokens;     /* P, tokens per partition */
  int32_t num_splits;       /* S = ceil(max_context_len / P) */
  int32_t variant;          /* 0 = CUDA-core kernel, 1 = mma.sync tensor-core
                               kernel, 2 = tcgen05 tensor-core kernel */
  int32_t warps_per_cta;
  int32_t stages_per_warp;
  int32_t grid_ctas;
  size_t workspace_bytes;   /* 0 when no partials are needed */
} pkv_plan;

/*
 * Set the split-KV workspace that decode calls on the current device use
 * when they are given a NULL workspace (the library never allocates device
 * memory itself).  dev_ptr: caller-owned memory of the current device,
 * 16-byte aligned, `bytes` long (size it with pkv_workspace_bytes for the
 * largest shape in use); the library keeps the pointer, not the memory, so
 * keep it alive until it is replaced or cleared.  NULL clears the setting.
 * PKV_ERR_INVALID for bytes == 0 or a pointer that is not memory of the
 * current device, PKV_ERR_ALIGN for a misaligned one.  Calls that use the
 * set workspace must not overlap on the GPU.
 */
int pkv_set_workspace(void* dev_ptr, size_t bytes);

/*
 * KV append (slot scatter).  For every token t in [0, num_tokens) with
 * s = slot_mapping[t] >= 0, and every kv head h:
 *     k_cache[s / bs][h][s % bs][:] = k[t][h][:]
 *     v_cache[s / bs][h][s % bs][:] = v[t][h][:]
 * A negative slot means "write nothing" (padding).  Bit-exact copy.
 *
 *   shape         uses num_kv_heads, head_dim, block_size, num_blocks, dtype
 *   k, v          [num_tokens, Hkv, D], 16-byte aligned
 *   slot_mapping  [num_tokens] int32
 *   k_cache, v_cache  [NB, Hkv, bs, D], 16-byte aligned
 * Slots >= NB * bs are skipped and set PKV_DEV_BAD_SLOT.  Two tokens with the
 * same non-negative slot race (undefined which one lands).  num_tokens == 0 is
 * a no-op.
 */
int pkv_kv_cache_append(const pkv_shape* shape, const void* k, const void* v,
                        const int32_t* slot_mapping, int32_t num_tokens,
                        void* k_cache, void* v_cache, pkv_stream_t stream);

/*
 * Paged single-token decode attention.  For every sequence i and query head h,
 * with g = h / (Hq / Hkv) and L = context_lens[i]:
 *     k_t = k_cache[block_tables[i][t / bs]][g][t % bs][:],  t in [0, L)
 *     out[i][h][:] = sum_t softmax_t(scale * q[i][h] . k_t) * v_t
 * (v_t likewise from v_cache).
 *
 *   q, out            [B, Hq, D], 16-byte aligned
 *   k_cache, v_cache  [NB, Hkv, bs, D], 16-byte aligned
 *   block_tables      [B, MB] int32; entries past ceil(L / bs) are never read
 *   context_lens      [B] int32, each in [1, max_context_len]; counts the token
 *                     appended in this step
 *   scale             softmax scale (typically 1 / sqrt(D))
 *   workspace         caller-owned device scratch for split-KV partials, at
 *                     least pkv_plan.workspace_bytes, 16-byte aligned; its
 *                     contents need no initialisation.  NULL takes the
 *                     workspace set for the current device with
 *                     pkv_set_workspace (and workspace_bytes is ignored).
 *                     Calls that share a workspace must not overlap on the
 *                     GPU.  PKV_ERR_WORKSPACE, enqueuing nothing, when the
 *                     call needs partials (workspace_bytes > 0 in its plan)
 *                     and the workspace is missing, misaligned or too small.
 * A sequence whose length is out of range is skipped (its out rows are left
 * unwritten); the partitions of a sequence that hold an out-of-range block id
 * skip their work (the bad blocks are never read), so that sequence's out
 * rows are undefined (left unwritten when it has a single partition).  Either
 * way the device error word is set.  B == 0 is a
 * no-op.
 */
int pkv_paged_attn_decode(const pkv_shape* shape, const void* q,
                          const void* k_cache, const void* v_cache,
                          const int32_t* block_tables,
                          const int32_t* context_lens, float scale, void* out,
                          void* workspace, size_t workspace_bytes,
                          pkv_stream_t stream);

/*
 * One continuous-batching decode step in one launch (the append fused into
 * the decode): for every sequence i, this step's token (k_new[i], v_new[i])
 * is written at position L - 1, i.e. slot
 *     block_tables[i][(L-1) / bs] * bs + (L-1) % bs,
 * then decode attention runs over all L = context_lens[i] tokens.  The result
 * equals pkv_kv_cache_append with that slot mapping followed by
 * pkv_paged_attn_decode, bit for bit, caches included.  Per-iteration
 * metadata update plus attention over the block table (third page,
 * "continuous batching" and "PagedAttention" sections).
 *
 *   k_new, v_new  [B, Hkv, D], 16-byte aligned
 *   other arguments as pkv_paged_attn_decode; k_cache and v_cache are written
 * The block that receives a sequence's new token must not be referenced by
 * another sequence of the batch (copy it first when a prefix block is shared).
 * Runs on every kernel variant (split_tokens as for pkv_paged_attn_decode).
 */
int pkv_decode_step(const pkv_shape* shape, const void* q, const void* k_new,
                    const void* v_new, void* k_cache, void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens,
                    float scale, void* out, void* workspace, size_t workspace_bytes,
                    pkv_stream_t stream);

/*
 * pkv_paged_attn_decode for callers that cannot allocate device memory.  The
 * pages have no counterpart to this call; it exists for callers that own all
 * device memory themselves (an engine that reserved HBM for its KV block pool
 * and offers no allocator) or cannot afford cudaMalloc on their decode path.
 * Same arguments, layouts and results as pkv_paged_attn_decode, minus the
 * workspace: the split-KV partials go to a fixed 64 MiB array inside the
 * library (held on every GPU that loads the library until the process exits).
 *  - Returns PKV_ERR_WORKSPACE, enqueuing nothing, when the call's partials
 *    (pkv_plan.workspace_bytes) exceed 64 MiB; raise split_tokens to fit.
 *  - The first call on a device looks up the array's address on that device;
 *    make that first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (nothing in it needs clearing): calls that overlap on the GPU
 *    race.  Never calls cudaMalloc, cudaFree or any allocating routine.
 */
int pkv_paged_attn_decode_noalloc(const pkv_shape* shape, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables,
                                  const int32_t* context_lens, float scale,
                                  void* out, pkv_stream_t stream);

/*
 * Whole-block copy between two pools of the same block shape: for i in
 * [0, num_pairs), block pairs[2i] of (src_k, src_v) is copied to block
 * pairs[2i+1] of (dst_k, dst_v), every kv head.  Serves copy-on-write inside
 * the GPU pool and the swap-out / swap-in of the tiered cache (first page,
 * section 4.2: cold blocks move to pinned CPU memory and come back by DMA).
 * Bit-exact.
 *
 *   shape        uses num_kv_heads, head_dim, block_size, dtype
 *   src_*, dst_* [num_blocks, Hkv, bs, D] pools, 16-byte aligned, readable /
 *                writable by the GPU: device memory, or pinned host memory
 *                (cudaHostAlloc / cudaMallocHost), which the GPU reaches
 *                through its host pointer under unified addressing
 *   pairs        [num_pairs][2] int32, device-readable
 * Pairs with an id outside its pool are skipped and set PKV_DEV_BAD_BLOCK_ID.
 * Destination blocks must be distinct and must not be sources in the same
 * call.  num_pairs == 0 is a no-op.
 */
int pkv_copy_blocks(const pkv_shape* shape, const void* src_k, const void* src_v,
                    int32_t src_num_blocks, void* dst_k, void* dst_v,
                    int32_t dst_num_blocks, const int32_t* pairs, int32_t num_pairs,
                    pkv_stream_t stream);

/*
 * Block manager (host only, no GPU calls): the bookkeeping side of the paged
 * cache (first page, section 4.2: fixed-size blocks handed out on demand,
 * allocate(seq, num_tokens) takes ceil(num_tokens / block_size) blocks; the
 * tiered variant keeps the last gpu_window blocks of a sequence on the GPU
 * and moves older ones to pinned CPU memory), updated between launches as
 * sequences join, grow and leave (third page, "continuous batching").
 * Sequences made by pkv_bm_fork share their parent's blocks (reference
 * counted); writing into a shared block first copies it (copy-on-write).
 * Every call is thread-safe and returns PKV_OK or a negative PKV_ERR_*;
 * a call that fails changes nothing.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_gpu_blocks GPU blocks and num_cpu_blocks CPU blocks of
 * block_size tokens.  Each pool's free list is a stack: initially ids come
 * out lowest first, later the most recently freed block is reused first.
 * NULL on bad sizes. */
pkv_block_manager* pkv_bm_create(int32_t num_gpu_blocks, int32_t num_cpu_blocks,
                                 int32_t block_size);
void pkv_bm_destroy(pkv_block_manager* m);

/* New sequence holding num_tokens tokens (ceil(num_tokens / bs) GPU blocks).
 * PKV_ERR_INVALID if seq_id exists, PKV_ERR_NO_BLOCKS if the pool is short. */
int pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id, int32_t num_tokens);

/* New sequence `child` sharing every block of `parent` (all on the GPU). */
int pkv_bm_fork(pkv_block_manager* m, int64_t parent, int64_t child);

/* Reserve the slot of the sequence's next token: *slot = block * bs + offset.
 * When that token lands in a block shared with another sequence, the
 * sequence first gets a fresh block: *copy_src / *copy_dst name the GPU
 * blocks to copy (pkv_copy_blocks) before writing; both are -1 otherwise. */
int pkv_bm_append_token(pkv_block_manager* m, int64_t seq_id, int32_t* slot,
                        int32_t* copy_src, int32_t* copy_dst);

/* Drop the sequence; blocks no other sequence references become free. */
int pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id);

/* Move the sequence's blocks older than its last gpu_window blocks (those on
 * the GPU and not shared) to the CPU pool.  Writes num_pairs (gpu id, cpu id)
 * pairs for pkv_copy_blocks (GPU pool -> CPU pool) into pairs[2 * max_pairs].
 * The GPU blocks are free again as soon as this returns: enqueue the copy
 * before any launch that may write into reused blocks (same stream). */
int pkv_bm_swap_out(pkv_block_manager* m, int64_t seq_id, int32_t gpu_window,
                    int32_t* pairs, int32_t max_pairs, int32_t* num_pairs);

/* Bring every CPU block of the sequence back to the GPU pool: (cpu id,
 * gpu id) pairs for pkv_copy_blocks (CPU pool -> GPU pool). */
int pkv_bm_swap_in(pkv_block_manager* m, int64_t seq_id, int32_t* pairs,
                   int32_t max_pairs, int32_t* num_pairs);

int pkv_bm_num_free(pkv_block_manager* m, int32_t* gpu_blocks, int32_t* cpu_blocks);

int pkv_bm_seq_info(pkv_block_manager* m, int64_t seq_id, int32_t* num_tokens,
                    int32_t* num_blocks, int32_t* num_cpu_blocks);

/* Fill a decode batch's host arrays: block_tables [n, max_blocks_per_seq]
 * (-1 past each sequence's blocks) and context_lens [n].  PKV_ERR_INVALID if
 * a sequence is unknown, has CPU-resident blocks, or needs more than
 * max_blocks_per_seq blocks. */
int pkv_bm_block_tables(pkv_block_manager* m, const int64_t* seq_ids, int32_t n,
                        int32_t max_blocks_per_seq, int32_t* block_tables,
                        int32_t* context_lens);

/* Validate `shape` and report how pkv_paged_attn_decode will run on the
 * current device (split size, kernel variant, workspace size).  Host only;
 * reads device attributes once. */
int pkv_decode_plan(const pkv_shape* shape, pkv_plan* plan);

/* pkv_decode_plan for a GB300-class device with `num_sms` SMs (> 0, else
 * PKV_ERR_INVALID), without touching any device: plans ahead of a device and
 * lets the split rule be checked on a host without a GPU.  pkv_decode_plan
 * equals this call with the current device's SM count. */
int pkv_decode_plan_for(const pkv_shape* shape, int32_t num_sms, pkv_plan* plan);

/* Workspace bytes pkv_paged_attn_decode needs for `shape` (0 if none). */
int pkv_workspace_bytes(const pkv_shape* shape, size_t* bytes);

/* Read and clear the device-side error word of the current device.
 * Synchronises `stream`.  *code receives a PKV_DEV_* value (first error since
 * the last read). */
int pkv_get_device_error(int32_t* code, pkv_stream_t stream);

/*
 * Self-test of the bounded waits every kernel uses.  One warp waits on an
 * mbarrier that nothing ever arrives on, with a limit of `limit_us`
 * microseconds (1 .. 1000000) instead of the kernels' 0.5 s, then gives up,
 * records PKV_DEV_TIMEOUT in the device error word and exits.  The context
 * stays usable.  It checks that a wait that runs out is reported to the host
 * rather than hanging the GPU; it never faults or traps.
 */
int pkv_selftest_wait_timeout(int32_t limit_us, pkv_stream_t stream);

/* Human-readable text for a PKV_ERR_* code (static storage). */
const char* pkv_strerror(int code);

/* Number of kernels this library has launched in this process so far. */
uint64_t pkv_launch_count(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
