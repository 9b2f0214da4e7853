// Instantiates the tcgen05 decode kernel (head_dim 128; block size 16 or 32;
// N = 16 or 32 padded query heads; binary16 or bfloat16).
#include <atomic>

#include "pkv_decode_tc.cuh"

namespace pkv {
namespace {

template <bool BF, int BS, int N>
cudaError_t launch_tc(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                      cudaStream_t stream) {
  constexpr int SMEM = TcLayout<N>::BYTES;
  static_assert(SMEM <= 227 * 1024, "tcgen05 kernel shared memory");
  auto kern = paged_decode_tc<BF, BS, N>;
  // the shared-memory limit is raised once per device (every time past 32)
  static std::atomic<unsigned> mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = dev < 32 ? 1u << dev : 0u;
  if (bit == 0 || !(mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    mask.fetch_or(bit, std::memory_order_release);
  }
  // programmatic launch: the grid may become resident while the previous
  // kernel of the stream finishes (the kernel waits for it before any access)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.Hkv * a.S);
  cfg.blockDim = dim3(TcLayout<N>::THREADS);
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

template <bool BF>
cudaError_t dispatch_tc(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                        int block_size, cudaStream_t stream) {
  const bool wide = a.G > 16;
  if (block_size == 16)
    return wide ? launch_tc<BF, 16, 32>(a, tk, tv, stream) : launch_tc<BF, 16, 16>(a, tk, tv, stream);
  if (block_size == 32)
    return wide ? launch_tc<BF, 32, 32>(a, tk, tv, stream) : launch_tc<BF, 32, 16>(a, tk, tv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                             bool bf16, int head_dim, int block_size, cudaStream_t stream) {
  if (head_dim != 128 || a.G < 1 || a.G > 32) return cudaErrorInvalidValue;
  return bf16 ? dispatch_tc<true>(a, tk, tv, block_size, stream)
              : dispatch_tc<false>(a, tk, tv, block_size, stream);
}

int tc_smem_bytes(int G) { return G > 16 ? TcLayout<32>::BYTES : TcLayout<16>::BYTES; }
int tc_ring_slots(int G) { return G > 16 ? TcLayout<32>::SLOTS : TcLayout<16>::SLOTS; }
int tc_warps(int G) { return (G > 16 ? TcLayout<32>::THREADS : TcLayout<16>::THREADS) / 32; }

}  // namespace pkv
