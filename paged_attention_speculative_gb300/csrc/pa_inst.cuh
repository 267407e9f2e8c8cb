// pa_inst.cuh — instantiation helper: info + launch for one head dim.
#pragma once

#include "pa_launch.h"
#include "pa_partition_mma.cuh"

namespace pa {

template <int D, int KV, int NT, bool GATHER = false>
MmaKernelInfo mma_info_t() {
  using S = MmaSmem<D, KV, NT, GATHER>;
  return MmaKernelInfo{MmaCfg<D, KV, GATHER>::SK, S::BYTES, S::CTAS_PER_SM};
}

template <int D, int KV, int NT, bool TREE, bool GATHER = false>
cudaError_t launch_mma_tt(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                          cudaStream_t st) {
  auto kern = pa_partition_mma<D, KV, NT, TREE, GATHER>;
  const int smem = MmaSmem<D, KV, NT, GATHER>::BYTES;
  // Raise the dynamic shared-memory limit once per process and device.
  static int configured_for[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !__atomic_load_n(&configured_for[dev], __ATOMIC_ACQUIRE)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    __atomic_store_n(&configured_for[dev], 1, __ATOMIC_RELEASE);
  }
  return launch_dependent(kern, grid, dim3(GATHER ? kThreads + 32 : kThreads), smem, st, k, v, a);
}

// Tree-mask verify runs its own instantiation, so the causal kernels keep
// their code.
template <int D, int KV, int NT, bool GATHER = false>
cudaError_t launch_mma_t(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                         cudaStream_t st) {
  return a.tree_mask != nullptr ? launch_mma_tt<D, KV, NT, true, GATHER>(k, v, a, grid, st)
                                : launch_mma_tt<D, KV, NT, false, GATHER>(k, v, a, grid, st);
}

}  // namespace pa

// Expands to the info / launch dispatchers of head dim D_ for the listed
// (kv, nt) combinations.
#define PA_DISPATCH_CASE(D_, KV_, NT_)                                   \
  if (kv == KV_ && nt == NT_) {                                          \
    if (ok) *ok = true;                                                  \
    return mma_info_t<D_, KV_, NT_>();                                   \
  }
#define PA_LAUNCH_CASE(D_, KV_, NT_) \
  if (kv == KV_ && nt == NT_) return launch_mma_t<D_, KV_, NT_>(k, v, a, grid, st);
