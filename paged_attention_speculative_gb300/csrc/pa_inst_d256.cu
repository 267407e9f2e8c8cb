// Tensor-core partition kernels for head_dim 256 (16-bit and u8 caches; one
// 8-row n-tile per warp keeps the 256-wide accumulator in registers).
#include "pa_inst.cuh"

namespace pa {

MmaKernelInfo mma_info_d256(int kv, int nt, bool* ok) {
  if (ok) *ok = false;
  PA_DISPATCH_CASE(256, KV_BF16, 1)
  PA_DISPATCH_CASE(256, KV_F16, 1)
  PA_DISPATCH_CASE(256, KV_U8, 1)
  return MmaKernelInfo{0, 0, 0};
}

cudaError_t launch_mma_d256(int kv, int nt, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                            cudaStream_t st) {
  PA_LAUNCH_CASE(256, KV_BF16, 1)
  PA_LAUNCH_CASE(256, KV_F16, 1)
  PA_LAUNCH_CASE(256, KV_U8, 1)
  return cudaErrorInvalidValue;
}

}  // namespace pa
