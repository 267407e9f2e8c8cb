// Tensor-core partition kernels for head_dim 128 (16-bit and u8 caches).
#include "pa_inst.cuh"

namespace pa {

MmaKernelInfo mma_info_d128(int kv, int nt, bool* ok) {
  if (ok) *ok = false;
  PA_DISPATCH_CASE(128, KV_BF16, 1)
  PA_DISPATCH_CASE(128, KV_BF16, 2)
  PA_DISPATCH_CASE(128, KV_F16, 1)
  PA_DISPATCH_CASE(128, KV_F16, 2)
  PA_DISPATCH_CASE(128, KV_U8, 1)
  PA_DISPATCH_CASE(128, KV_U8, 2)
  return MmaKernelInfo{0, 0, 0};
}

cudaError_t launch_mma_d128(int kv, int nt, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                            cudaStream_t st) {
  PA_LAUNCH_CASE(128, KV_BF16, 1)
  PA_LAUNCH_CASE(128, KV_BF16, 2)
  PA_LAUNCH_CASE(128, KV_F16, 1)
  PA_LAUNCH_CASE(128, KV_F16, 2)
  PA_LAUNCH_CASE(128, KV_U8, 1)
  PA_LAUNCH_CASE(128, KV_U8, 2)
  return cudaErrorInvalidValue;
}

}  // namespace pa
