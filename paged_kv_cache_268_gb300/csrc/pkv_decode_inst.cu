// Instantiates the decode kernels for one element type and one compute
// variant; compiled once per (PKV_INST_BF16, PKV_INST_MMA) pair.
#include <atomic>

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

// Raise a kernel's dynamic shared-memory limit once per device (every time
// on devices past the 32 the mask tracks).  Threads that race here both set
// the same attribute, which is harmless.
template <class K>
cudaError_t configure(K kern, int smem, std::atomic<unsigned>* mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = dev < 32 ? 1u << dev : 0u;
  if (bit == 0 || !(mask->load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mask->fetch_or(bit, std::memory_order_release);
  }
  return cudaSuccess;
}

template <int D, int BS, class Compute>
cudaError_t launch_one(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  constexpr int NW = geo_warps(D, BS);
  constexpr int NS = part_stages(D, BS, Compute::NH);
  constexpr int SMEM = part_smem(D, BS, Compute::NH);
  auto kern = paged_decode_kernel<kBF, D, BS, NW, NS, Compute>;
  static std::atomic<unsigned> mask{0};
  cudaError_t e = configure(kern, SMEM, &mask);
  if (e != cudaSuccess) return e;
  // programmatic launch: the grid may become resident while the previous
  // kernel of the stream finishes (the kernel waits for it before any access)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.Hkv * a.S);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, tk, tv);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, int BS>
cudaError_t launch_variant(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t stream) {
#if PKV_INST_MMA
  if (a.G >= 1 && a.G <= 8)
    return launch_one<D, BS, MmaCompute<kBF, D, BS, 1>>(a, tk, tv, stream);
  if (a.G >= 9 && a.G <= 16)
    return launch_one<D, BS, MmaCompute<kBF, D, BS, 2>>(a, tk, tv, stream);
  if (a.G >= 17 && a.G <= 32)
    return launch_one<D, BS, MmaCompute<kBF, D, BS, 4>>(a, tk, tv, stream);
#else
  if (a.G == 1)
    return launch_one<D, BS, SimtCompute<kBF, D, BS, 1>>(a, tk, tv, stream);
  if (a.G == 2)
    return launch_one<D, BS, SimtCompute<kBF, D, BS, 2>>(a, tk, tv, stream);
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
