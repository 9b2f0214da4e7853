/*
 * The C ABI driven from a plain C11 program: no C++, no PyTorch, no binding.
 * Device buffers come from cudaMalloc, every call goes through include/pkv.h,
 * results are copied back and compared with the fp64 oracle (linked in from
 * the oracle's C source; test infrastructure, like this program).
 *
 * Checked, on one seeded batch with ragged lengths (1 token, exactly one
 * block, one block and a token, several partitions, a ragged tail):
 *   - pkv_kv_cache_append: caches bit-identical to the oracle's append, with a
 *     padding token (slot -1) that must write nothing;
 *   - pkv_paged_attn_decode with a caller workspace: every element within the
 *     tolerance of the oracle's attention over the appended caches;
 *   - the same call with the workspace set by pkv_set_workspace and NULL
 *     passed, and pkv_paged_attn_decode_noalloc: bit-identical outputs;
 *   - pkv_decode_step from the caches before the append: outputs and caches
 *     bit-identical to append followed by decode;
 *   - host-side argument errors return their codes and enqueue nothing, and
 *     the device error word stays clear.
 *
 * Usage: decode_c <dtype 0|1> <kernel> <split_tokens> <group>, where group is
 * Hq / Hkv (two kv heads).  Prints one line
 * "OK variant=<v> splits=<S>" and exits 0 when every check passes; otherwise
 * prints what failed and exits 1.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pkv.h"

/* the oracle's C entry points */
int pkv_oracle_decode(int B, int Hq, int Hkv, int D, int bs, int NB, int MB, int dtype,
                      const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      double scale, double* out);
int pkv_oracle_append(int T, int Hkv, int D, int bs, int NB, const uint16_t* k,
                      const uint16_t* v, const int32_t* slot_mapping,
                      uint16_t* k_cache, uint16_t* v_cache);
double pkv_oracle_half_to_double(uint16_t h);
double pkv_oracle_bf16_to_double(uint16_t h);

static int failures = 0;

#define CHECK(cond, ...)                                   \
  do {                                                     \
    if (!(cond)) {                                         \
      fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      fprintf(stderr, __VA_ARGS__);                        \
      fprintf(stderr, "\n");                               \
      ++failures;                                          \
    }                                                      \
  } while (0)

#define CUDA(call)                                                           \
  do {                                                                       \
    cudaError_t e_ = (call);                                                 \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_),    \
              __FILE__, __LINE__);                                           \
      exit(1);                                                               \
    }                                                                        \
  } while (0)

/* splitmix64: a counter-based generator, one 64-bit output per counter. */
static uint64_t mix(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

/* The 16-bit pattern of m / 128 for |m| < 128, built from the two formats'
 * field layouts (sign, biased exponent, fraction); exact in both. */
static uint16_t encode(int m, int dtype) {
  if (m == 0) return 0;
  uint16_t sign = m < 0 ? 0x8000u : 0u;
  int a = m < 0 ? -m : m, e = 0;
  while ((2 << e) <= a) ++e;                 /* 2^e <= a < 2^(e+1) */
  int frac = a - (1 << e);
  if (dtype == PKV_F16)
    return (uint16_t)(sign | ((e - 7 + 15) << 10) | (frac << (10 - e)));
  return (uint16_t)(sign | ((e - 7 + 127) << 7) | (frac << (7 - e)));
}

static void fill(uint16_t* x, size_t n, uint64_t stream, int dtype) {
  for (size_t i = 0; i < n; ++i)
    x[i] = encode((int)(mix(stream * 0x100000000ull + i) % 255) - 127, dtype);
}

static void* dalloc(size_t bytes) {
  void* p = NULL;
  CUDA(cudaMalloc(&p, bytes ? bytes : 16));
  return p;
}

static void h2d(void* d, const void* h, size_t bytes) {
  CUDA(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
}

static void d2h(void* h, const void* d, size_t bytes) {
  CUDA(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
}

int main(int argc, char** argv) {
  if (argc != 5) {
    fprintf(stderr, "usage: %s <dtype 0|1> <kernel> <split_tokens> <group>\n", argv[0]);
    return 2;
  }
  const int dtype = atoi(argv[1]), kernel = atoi(argv[2]), split = atoi(argv[3]);
  const int Hkv = 2, Hq = Hkv * atoi(argv[4]);
  double (*widen)(uint16_t) = dtype == PKV_F16 ? pkv_oracle_half_to_double
                                               : pkv_oracle_bf16_to_double;

  /* the encoder, checked against the oracle's converters */
  for (int m = -127; m <= 127; ++m)
    CHECK(widen(encode(m, dtype)) == m / 128.0, "encode(%d) widens to %.17g", m,
          widen(encode(m, dtype)));

  enum { B = 6, D = 128, BS = 16 };
  const int32_t lens[B] = {1, 16, 17, 333, 2048, 2600};
  int MB = 0, used = 0;
  for (int i = 0; i < B; ++i) {
    int nb = (lens[i] + BS - 1) / BS;
    used += nb;
    if (nb > MB) MB = nb;
  }
  const int NB = used + 7;                   /* spare blocks nobody reads */
  const size_t per_tok = (size_t)Hkv * D, cache_n = (size_t)NB * Hkv * BS * D;
  const size_t q_n = (size_t)B * Hq * D;
  const float scale = 0.08838834764831845f; /* 1 / sqrt(128) */

  /* physical ids: a seeded permutation of [0, NB), handed out in order */
  int32_t* perm = malloc(sizeof(int32_t) * NB);
  for (int i = 0; i < NB; ++i) perm[i] = i;
  for (int i = NB - 1; i > 0; --i) {
    int j = (int)(mix(0x5eedull + (uint64_t)i) % (uint64_t)(i + 1));
    int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
  }
  int32_t* tables = calloc((size_t)B * MB, sizeof(int32_t));
  for (int i = 0, next = 0; i < B; ++i) {
    for (int j = 0; j < MB; ++j)
      tables[i * MB + j] = j < (lens[i] + BS - 1) / BS ? perm[next++] : -1;
  }

  uint16_t* q = malloc(q_n * 2);
  uint16_t* kc0 = malloc(cache_n * 2);
  uint16_t* vc0 = malloc(cache_n * 2);
  uint16_t* kc = malloc(cache_n * 2);
  uint16_t* vc = malloc(cache_n * 2);
  uint16_t* got_k = malloc(cache_n * 2);
  uint16_t* got_v = malloc(cache_n * 2);
  fill(q, q_n, 1, dtype);
  fill(kc0, cache_n, 2, dtype);
  fill(vc0, cache_n, 3, dtype);

  /* this step's tokens: one per sequence at position L - 1, and one padding
   * token (slot -1) that must write nothing */
  const int T = B + 1;
  uint16_t* kn = malloc((size_t)T * per_tok * 2);
  uint16_t* vn = malloc((size_t)T * per_tok * 2);
  fill(kn, (size_t)T * per_tok, 4, dtype);
  fill(vn, (size_t)T * per_tok, 5, dtype);
  int32_t slots[B + 1];
  for (int i = 0; i < B; ++i)
    slots[i] = tables[i * MB + (lens[i] - 1) / BS] * BS + (lens[i] - 1) % BS;
  slots[B] = -1;

  /* the oracle: append, then attention over the appended caches */
  memcpy(kc, kc0, cache_n * 2);
  memcpy(vc, vc0, cache_n * 2);
  CHECK(pkv_oracle_append(T, Hkv, D, BS, NB, kn, vn, slots, kc, vc) == 0, "oracle append");
  double* ref = malloc(sizeof(double) * q_n);
  CHECK(pkv_oracle_decode(B, Hq, Hkv, D, BS, NB, MB, dtype, q, kc, vc, tables, lens,
                          (double)scale, ref) == 0, "oracle decode");

  cudaStream_t st;
  CUDA(cudaStreamCreate(&st));
  pkv_stream_t s = (pkv_stream_t)st;
  void *d_q = dalloc(q_n * 2), *d_kc = dalloc(cache_n * 2), *d_vc = dalloc(cache_n * 2);
  void *d_kn = dalloc((size_t)T * per_tok * 2), *d_vn = dalloc((size_t)T * per_tok * 2);
  void *d_tab = dalloc(sizeof(int32_t) * B * MB), *d_len = dalloc(sizeof(lens));
  void *d_slot = dalloc(sizeof(slots)), *d_out = dalloc(q_n * 2);
  h2d(d_q, q, q_n * 2);
  h2d(d_kc, kc0, cache_n * 2);
  h2d(d_vc, vc0, cache_n * 2);
  h2d(d_kn, kn, (size_t)T * per_tok * 2);
  h2d(d_vn, vn, (size_t)T * per_tok * 2);
  h2d(d_tab, tables, sizeof(int32_t) * B * MB);
  h2d(d_len, lens, sizeof(lens));
  h2d(d_slot, slots, sizeof(slots));

  pkv_shape sh = {B, Hq, Hkv, D, BS, NB, MB, lens[B - 1], dtype, split, kernel};
  pkv_plan plan;
  size_t ws_bytes = 0;
  int rc = pkv_decode_plan(&sh, &plan);
  if (rc != PKV_OK) {
    fprintf(stderr, "pkv_decode_plan: %s\n", pkv_strerror(rc));
    return 1;
  }
  CHECK(pkv_workspace_bytes(&sh, &ws_bytes) == PKV_OK && ws_bytes == plan.workspace_bytes,
        "workspace bytes %zu vs plan %zu", ws_bytes, plan.workspace_bytes);
  void* d_ws = dalloc(ws_bytes);
  const uint64_t launches0 = pkv_launch_count();

  /* host-side argument errors: codes returned, nothing enqueued */
  CHECK(pkv_paged_attn_decode(NULL, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, d_ws,
                              ws_bytes, s) == PKV_ERR_NULL, "NULL shape");
  pkv_shape bad = sh;
  bad.num_q_heads = 7;
  CHECK(pkv_paged_attn_decode(&bad, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, d_ws,
                              ws_bytes, s) == PKV_ERR_INVALID, "Hq %% Hkv != 0");
  CHECK(pkv_paged_attn_decode(&sh, (const char*)d_q + 2, d_kc, d_vc, d_tab, d_len, scale,
                              d_out, d_ws, ws_bytes, s) == PKV_ERR_ALIGN, "misaligned q");
  if (ws_bytes > 0)
    CHECK(pkv_paged_attn_decode(&sh, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, d_ws,
                                ws_bytes - 16, s) == PKV_ERR_WORKSPACE, "short workspace");
  CHECK(pkv_launch_count() == launches0, "a rejected call launched a kernel");

  /* append, then decode with the caller's workspace */
  rc = pkv_kv_cache_append(&sh, d_kn, d_vn, d_slot, T, d_kc, d_vc, s);
  CHECK(rc == PKV_OK, "append: %s", pkv_strerror(rc));
  rc = pkv_paged_attn_decode(&sh, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, d_ws,
                             ws_bytes, s);
  CHECK(rc == PKV_OK, "decode: %s", pkv_strerror(rc));
  CUDA(cudaStreamSynchronize(st));
  d2h(got_k, d_kc, cache_n * 2);
  d2h(got_v, d_vc, cache_n * 2);
  CHECK(memcmp(got_k, kc, cache_n * 2) == 0 && memcmp(got_v, vc, cache_n * 2) == 0,
        "appended caches differ from the oracle's");
  uint16_t* out1 = malloc(q_n * 2);
  d2h(out1, d_out, q_n * 2);
  int out_of_tol = 0;
  double worst = 0.0;
  for (size_t e = 0; e < q_n; ++e) {
    double g = widen(out1[e]), err = fabs(g - ref[e]);
    double bound = 2e-3 + 1e-2 * fabs(ref[e]);   /* the Python parity tests' bound */
    if (!(err <= bound)) ++out_of_tol;
    if (err > worst) worst = err;
  }
  CHECK(out_of_tol == 0, "%d of %zu elements out of tolerance (worst |err| %.3g)",
        out_of_tol, q_n, worst);

  /* the set workspace, then the no-alloc call: the same bits */
  uint16_t* out2 = malloc(q_n * 2);
  CHECK(pkv_set_workspace(d_ws, ws_bytes ? ws_bytes : 16) == PKV_OK, "set workspace");
  CUDA(cudaMemset(d_out, 0, q_n * 2));
  rc = pkv_paged_attn_decode(&sh, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, NULL, 0, s);
  CHECK(rc == PKV_OK, "decode with the set workspace: %s", pkv_strerror(rc));
  CUDA(cudaStreamSynchronize(st));
  d2h(out2, d_out, q_n * 2);
  CHECK(memcmp(out1, out2, q_n * 2) == 0, "set-workspace output differs");
  CHECK(pkv_set_workspace(NULL, 0) == PKV_OK, "clear workspace");
  if (ws_bytes > 0)
    CHECK(pkv_paged_attn_decode(&sh, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, NULL, 0,
                                s) == PKV_ERR_WORKSPACE, "cleared workspace still used");

  CUDA(cudaMemset(d_out, 0, q_n * 2));
  rc = pkv_paged_attn_decode_noalloc(&sh, d_q, d_kc, d_vc, d_tab, d_len, scale, d_out, s);
  CHECK(rc == PKV_OK, "no-alloc decode: %s", pkv_strerror(rc));
  CUDA(cudaStreamSynchronize(st));
  d2h(out2, d_out, q_n * 2);
  CHECK(memcmp(out1, out2, q_n * 2) == 0, "no-alloc output differs");

  /* the fused step from the caches as they were before the append */
  h2d(d_kc, kc0, cache_n * 2);
  h2d(d_vc, vc0, cache_n * 2);
  CUDA(cudaMemset(d_out, 0, q_n * 2));
  rc = pkv_decode_step(&sh, d_q, d_kn, d_vn, d_kc, d_vc, d_tab, d_len, scale, d_out, d_ws,
                       ws_bytes, s);
  CHECK(rc == PKV_OK, "fused step: %s", pkv_strerror(rc));
  CUDA(cudaStreamSynchronize(st));
  d2h(out2, d_out, q_n * 2);
  d2h(got_k, d_kc, cache_n * 2);
  d2h(got_v, d_vc, cache_n * 2);
  CHECK(memcmp(out1, out2, q_n * 2) == 0, "fused step output differs from append + decode");
  CHECK(memcmp(got_k, kc, cache_n * 2) == 0 && memcmp(got_v, vc, cache_n * 2) == 0,
        "fused step caches differ from the oracle's append");

  int32_t code = -1;
  CHECK(pkv_get_device_error(&code, s) == PKV_OK && code == PKV_DEV_OK,
        "device error word %d", (int)code);
  CHECK(pkv_launch_count() > launches0, "no kernel launched");

  CUDA(cudaStreamDestroy(st));
  void* dev[] = {d_q, d_kc, d_vc, d_kn, d_vn, d_tab, d_len, d_slot, d_out, d_ws};
  for (size_t i = 0; i < sizeof(dev) / sizeof(dev[0]); ++i) CUDA(cudaFree(dev[i]));
  free(perm); free(tables); free(q); free(kc0); free(vc0); free(kc); free(vc);
  free(got_k); free(got_v); free(kn); free(vn); free(ref); free(out1); free(out2);

  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("OK variant=%d splits=%d\n", plan.variant, plan.num_splits);
  return 0;
}
