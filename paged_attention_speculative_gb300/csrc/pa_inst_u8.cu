// pa_inst_u8.cu — instantiations and launcher of the u8 tensor-memory
// partition kernel (row tiles 16 / 32, pages of 16 / 32 / 64 tokens).
#include "pa_launch.h"
#include "pa_partition_u8.cuh"

namespace pa {

namespace {
template <int N, int PS>
cudaError_t launch_u8_t(const CUtensorMap& k, const PartArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = pa_partition_u8<N, PS>;
  const int smem = U8Cfg<N, PS>::BYTES;
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !__atomic_load_n(&configured_for[dev], __ATOMIC_ACQUIRE)) {
    if constexpr (U8Cfg<N, PS>::kRegSplit) {
      // the warpgroups' register targets are sized for this pool: a kernel
      // built with fewer registers per thread would wait forever in the
      // increase, so it is never launched
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs < U8Cfg<N, PS>::kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    __atomic_store_n(&configured_for[dev], 1, __ATOMIC_RELEASE);
  }
  return launch_dependent(kern, grid, dim3(640), smem, st, k, a);
}

template <int N>
cudaError_t launch_u8_n(int ps, const CUtensorMap& k, const PartArgs& a, dim3 grid, cudaStream_t st) {
  if (ps == 16) return launch_u8_t<N, 16>(k, a, grid, st);
  if (ps == 32) return launch_u8_t<N, 32>(k, a, grid, st);
  if (ps == 64) return launch_u8_t<N, 64>(k, a, grid, st);
  return cudaErrorInvalidValue;
}
}  // namespace

MmaKernelInfo u8_info(int n, int ps, bool* ok) {
  *ok = (n == 16 || n == 32) && (ps == 16 || ps == 32 || ps == 64);
  if (!*ok) return MmaKernelInfo{0, 0, 0};
  int bytes = 0;
  if (n == 16) bytes = ps == 16 ? U8Cfg<16, 16>::BYTES : (ps == 32 ? U8Cfg<16, 32>::BYTES : U8Cfg<16, 64>::BYTES);
  else bytes = ps == 16 ? U8Cfg<32, 16>::BYTES : (ps == 32 ? U8Cfg<32, 32>::BYTES : U8Cfg<32, 64>::BYTES);
  return MmaKernelInfo{128, bytes, 1};
}

cudaError_t launch_u8(int n, int ps, const CUtensorMap& k, const PartArgs& a, dim3 grid, cudaStream_t st) {
  if (n == 16) return launch_u8_n<16>(ps, k, a, grid, st);
  if (n == 32) return launch_u8_n<32>(ps, k, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
