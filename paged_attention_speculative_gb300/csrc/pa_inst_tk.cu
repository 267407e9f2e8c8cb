// Tensor-memory partition kernels with the keys on the MMA's M dimension.
#include "pa_launch.h"
#include "pa_partition_tk.cuh"
#include "pa_partition_tku8.cuh"

namespace pa {

namespace {
template <int D, int KV, int N>
cudaError_t launch_tk_t(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = pa_partition_tk<D, KV, N>;
  const int smem = TkCfg<D, KV, N>::BYTES;
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !__atomic_load_n(&configured_for[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    __atomic_store_n(&configured_for[dev], 1, __ATOMIC_RELEASE);
  }
  return launch_dependent(kern, grid, dim3(192), smem, st, k, v, a);
}

template <int D, int KV>
cudaError_t launch_tk_n(int n, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                        cudaStream_t st) {
  if (n == 16) return launch_tk_t<D, KV, 16>(k, v, a, grid, st);
  if (n == 32) return launch_tk_t<D, KV, 32>(k, v, a, grid, st);
  if (n == 64) return launch_tk_t<D, KV, 64>(k, v, a, grid, st);
  return cudaErrorInvalidValue;
}
template <int N>
cudaError_t launch_tku8_t(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = pa_partition_tku8<N>;
  const int smem = TkU8Cfg<N>::BYTES;
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !__atomic_load_n(&configured_for[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    __atomic_store_n(&configured_for[dev], 1, __ATOMIC_RELEASE);
  }
  return launch_dependent(kern, grid, dim3(320), smem, st, k, v, a);
}
}  // namespace

MmaKernelInfo tku8_info(int n, bool* ok) {
  *ok = (n == 16 || n == 32);
  if (!*ok) return MmaKernelInfo{0, 0, 0};
  return MmaKernelInfo{TkU8Cfg<16>::HK, n == 16 ? TkU8Cfg<16>::BYTES : TkU8Cfg<32>::BYTES, 1};
}

cudaError_t launch_tku8(int n, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                        cudaStream_t st) {
  if (n == 16) return launch_tku8_t<16>(k, v, a, grid, st);
  if (n == 32) return launch_tku8_t<32>(k, v, a, grid, st);
  return cudaErrorInvalidValue;
}

MmaKernelInfo tk_info(int D, int kv, int n, bool* ok) {
  *ok = (D == 64 || D == 128) && (kv == KV_BF16 || kv == KV_F16) && (n == 16 || n == 32 || n == 64);
  if (!*ok) return MmaKernelInfo{0, 0, 0};
  int bytes = 0;
  if (D == 64) bytes = n == 16 ? TkCfg<64, KV_BF16, 16>::BYTES : (n == 32 ? TkCfg<64, KV_BF16, 32>::BYTES : TkCfg<64, KV_BF16, 64>::BYTES);
  else bytes = n == 16 ? TkCfg<128, KV_BF16, 16>::BYTES : (n == 32 ? TkCfg<128, KV_BF16, 32>::BYTES : TkCfg<128, KV_BF16, 64>::BYTES);
  return MmaKernelInfo{128, bytes, 1};
}

cudaError_t launch_tk(int D, int kv, int n, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                      cudaStream_t st) {
  if (D == 64 && kv == KV_BF16) return launch_tk_n<64, KV_BF16>(n, k, v, a, grid, st);
  if (D == 64 && kv == KV_F16) return launch_tk_n<64, KV_F16>(n, k, v, a, grid, st);
  if (D == 128 && kv == KV_BF16) return launch_tk_n<128, KV_BF16>(n, k, v, a, grid, st);
  if (D == 128 && kv == KV_F16) return launch_tk_n<128, KV_F16>(n, k, v, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
