// Tensor-memory (tcgen05) partition kernels for pages of 1, 2 or 4 tokens:
// the cp.async-gather producer, head_dim 64 / 128, bf16 / f16 caches.
#include "pa_inst_tc.cuh"

namespace pa {

namespace {
template <int D, int KV>
cudaError_t launch_g(const PartArgs& a, dim3 grid, cudaStream_t st) {
  CUtensorMap unused;  // the gather producer reads the caches through plain pointers
  memset(&unused, 0, sizeof(unused));
  return a.tree_mask != nullptr ? launch_tc_tt<D, KV, true, true>(unused, unused, a, grid, st)
                                : launch_tc_tt<D, KV, false, true>(unused, unused, a, grid, st);
}
}  // namespace

cudaError_t launch_tc_gather(int D, int kv, const PartArgs& a, dim3 grid, cudaStream_t st) {
  if (D == 64 && kv == KV_BF16) return launch_g<64, KV_BF16>(a, grid, st);
  if (D == 64 && kv == KV_F16) return launch_g<64, KV_F16>(a, grid, st);
  if (D == 128 && kv == KV_BF16) return launch_g<128, KV_BF16>(a, grid, st);
  if (D == 128 && kv == KV_F16) return launch_g<128, KV_F16>(a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
