// Prefill tile kernels of a mixed batch (tcgen05): head_dim 64 / 128, bf16 / f16 caches.
#include "pa_combine.cuh"
#include "pa_launch.h"
#include "pa_prefill_tc.cuh"

namespace pa {

namespace {
template <int D, int KV, bool SPLIT>
cudaError_t launch_p(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = pa_prefill_tc<D, KV, SPLIT>;
  const int smem = PfCfg<D, KV>::BYTES;
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

cudaError_t launch_prefill_tc(int D, int kv, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a,
                              dim3 grid, cudaStream_t st) {
  const bool split = grid.z > 1;
  if (D == 64 && kv == KV_BF16)
    return split ? launch_p<64, KV_BF16, true>(k, v, a, grid, st) : launch_p<64, KV_BF16, false>(k, v, a, grid, st);
  if (D == 64 && kv == KV_F16)
    return split ? launch_p<64, KV_F16, true>(k, v, a, grid, st) : launch_p<64, KV_F16, false>(k, v, a, grid, st);
  if (D == 128 && kv == KV_BF16)
    return split ? launch_p<128, KV_BF16, true>(k, v, a, grid, st) : launch_p<128, KV_BF16, false>(k, v, a, grid, st);
  if (D == 128 && kv == KV_F16)
    return split ? launch_p<128, KV_F16, true>(k, v, a, grid, st) : launch_p<128, KV_F16, false>(k, v, a, grid, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_combine(int D, const CombineArgs& a, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.total_tokens) * a.Hq;
  const dim3 grid(static_cast<unsigned>((rows + 3) / 4));
  if (D == 64) return launch_dependent(pa_prefill_combine<64>, grid, dim3(128), 0, st, a);
  if (D == 128) return launch_dependent(pa_prefill_combine<128>, grid, dim3(128), 0, st, a);
  return cudaErrorInvalidValue;
}

}  // namespace pa
