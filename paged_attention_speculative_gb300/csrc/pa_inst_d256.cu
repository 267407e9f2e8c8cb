// Tensor-core partition kernels for head_dim 256 (16-bit and u8 caches; one
// 8-row n-tile per warp keeps the 256-wide accumulator in registers), and the
// 16-bit ones for pages of fewer than 8 tokens.
#include <cstring>

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

// Pages of 1, 2 or 4 tokens, 16-bit caches: the per-key bulk-copy producer
// (no tensor maps; the kernel's map parameters are left unread).
MmaKernelInfo mma_info_d256_gather(int kv, bool* ok) {
  *ok = kv == KV_BF16 || kv == KV_F16;
  return *ok ? (kv == KV_BF16 ? mma_info_t<256, KV_BF16, 1, true>() : mma_info_t<256, KV_F16, 1, true>())
             : MmaKernelInfo{0, 0, 0};
}

cudaError_t launch_mma_d256_gather(int kv, const PartArgs& a, dim3 grid, cudaStream_t st) {
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  if (kv == KV_BF16) return launch_mma_t<256, KV_BF16, 1, true>(unused, unused, a, grid, st);
  if (kv == KV_F16) return launch_mma_t<256, KV_F16, 1, true>(unused, unused, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
