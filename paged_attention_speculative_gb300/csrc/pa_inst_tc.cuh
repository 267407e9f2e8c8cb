// pa_inst_tc.cuh — launcher of one pa_partition_tc instantiation, shared by
// the units that instantiate the TMA and the cp.async-gather variants.
#pragma once

#include "pa_launch.h"
#include "pa_partition_tc.cuh"

namespace pa {

template <int D, int KV, bool TREE, bool GATHER>
cudaError_t launch_tc_tt(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid, cudaStream_t st) {
  auto kern = pa_partition_tc<D, KV, TREE, GATHER>;
  const int smem = TcCfg<D, KV>::BYTES;
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !__atomic_load_n(&configured_for[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    __atomic_store_n(&configured_for[dev], 1, __ATOMIC_RELEASE);
  }
  return launch_dependent(kern, grid, dim3(GATHER ? 128 + 32 * kGatherWarps : 128), smem, st, k, v, a);
}

}  // namespace pa
