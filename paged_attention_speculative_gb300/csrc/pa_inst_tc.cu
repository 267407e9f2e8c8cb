// Tensor-memory (tcgen05) partition kernels: head_dim 64 / 128, bf16 / f16 caches.
#include "pa_launch.h"
#include "pa_partition_tc.cuh"
#include "pa_inst_tc.cuh"

namespace pa {

namespace {
template <int D, int KV>
cudaError_t launch_tc_t(const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid, cudaStream_t st) {
  if (a.ps < kGatherBelowPageSize) return launch_tc_gather(D, KV, a, grid, st);
  return a.tree_mask != nullptr ? launch_tc_tt<D, KV, true, false>(k, v, a, grid, st)
                                : launch_tc_tt<D, KV, false, false>(k, v, a, grid, st);
}
}  // namespace

MmaKernelInfo tc_info(int D, int kv, bool* ok) {
  *ok = true;
  if (D == 64 && kv == KV_BF16) return MmaKernelInfo{TcCfg<64, KV_BF16>::SK, TcCfg<64, KV_BF16>::BYTES, 1};
  if (D == 64 && kv == KV_F16) return MmaKernelInfo{TcCfg<64, KV_F16>::SK, TcCfg<64, KV_F16>::BYTES, 1};
  if (D == 128 && kv == KV_BF16) return MmaKernelInfo{TcCfg<128, KV_BF16>::SK, TcCfg<128, KV_BF16>::BYTES, 1};
  if (D == 128 && kv == KV_F16) return MmaKernelInfo{TcCfg<128, KV_F16>::SK, TcCfg<128, KV_F16>::BYTES, 1};
  *ok = false;
  return MmaKernelInfo{0, 0, 0};
}

cudaError_t launch_tc(int D, int kv, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                      cudaStream_t st) {
  if (D == 64 && kv == KV_BF16) return launch_tc_t<64, KV_BF16>(k, v, a, grid, st);
  if (D == 64 && kv == KV_F16) return launch_tc_t<64, KV_F16>(k, v, a, grid, st);
  if (D == 128 && kv == KV_BF16) return launch_tc_t<128, KV_BF16>(k, v, a, grid, st);
  if (D == 128 && kv == KV_F16) return launch_tc_t<128, KV_F16>(k, v, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
