// Instantiates the decode kernels for one element type and one compute
// variant; compiled once per (PKV_INST_BF16, PKV_INST_MMA) pair.
#include "pkv_decode.cuh"

#ifndef PKV_INST_BF16
#error "define PKV_INST_BF16 (0 = binary16, 1 = bfloat16)"
#endif
#ifndef PKV_INST_MMA
#error "define PKV_INST_MMA (0 = CUDA-core variant, 1 = tensor-core variant)"
#endif

namespace pkv {
namespace {

constexpr bool kBF = PKV_INST_BF16 != 0;

template <int D, int BS, class Compute>
cudaError_t launch_one(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  constexpr int NW = geo_warps(D, BS);
  constexpr int NS = geo_stages(D, BS);
  constexpr int SMEM = geo_smem(D, BS);
  static_assert(NW * Compute::NH * (D + 2) * 4 <= NW * NS * stage_bytes(D, BS),
                "merge area must fit in the stage ring");
  auto kern = paged_decode_kernel<kBF, D, BS, NW, NS, Compute>;
  static int configured_mask = 0;  // one bit per device ordinal (< 32)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 32 && !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured_mask |= 1 << dev;
  }
  const unsigned grid = static_cast<unsigned>(a.B) * a.Hkv * a.S;
  kern<<<grid, NW * 32, SMEM, stream>>>(a, tk, tv);
  return cudaGetLastError();
}

template <int D, int BS>
cudaError_t launch_variant(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
#if PKV_INST_MMA
  if (a.G >= 3 && a.G <= 8) return launch_one<D, BS, MmaCompute<kBF, D, BS>>(a, tk, tv, stream);
#else
  if (a.G == 1) return launch_one<D, BS, SimtCompute<kBF, D, BS, 1>>(a, tk, tv, stream);
  if (a.G == 2) return launch_one<D, BS, SimtCompute<kBF, D, BS, 2>>(a, tk, tv, stream);
#endif
  return cudaErrorInvalidValue;
}

cudaError_t dispatch(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int D,
                     int BS, cudaStream_t stream) {
  if (D == 64 && BS == 16) return launch_variant<64, 16>(a, tk, tv, stream);
  if (D == 64 && BS == 32) return launch_variant<64, 32>(a, tk, tv, stream);
  if (D == 128 && BS == 16) return launch_variant<128, 16>(a, tk, tv, stream);
  if (D == 128 && BS == 32) return launch_variant<128, 32>(a, tk, tv, stream);
  if (D == 256 && BS == 16) return launch_variant<256, 16>(a, tk, tv, stream);
  if (D == 256 && BS == 32) return launch_variant<256, 32>(a, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

#if PKV_INST_BF16 && PKV_INST_MMA
#define PKV_LAUNCH_NAME launch_decode_bf16_mma
#elif PKV_INST_BF16
#define PKV_LAUNCH_NAME launch_decode_bf16_simt
#elif PKV_INST_MMA
#define PKV_LAUNCH_NAME launch_decode_f16_mma
#else
#define PKV_LAUNCH_NAME launch_decode_f16_simt
#endif

cudaError_t PKV_LAUNCH_NAME(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                            int head_dim, int block_size, cudaStream_t stream) {
  return dispatch(a, tk, tv, head_dim, block_size, stream);
}

}  // namespace pkv
