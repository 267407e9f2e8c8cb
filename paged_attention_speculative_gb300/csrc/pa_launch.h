// pa_launch.h — host-side launch helpers shared by the C-ABI implementation
// and the per-head-dim instantiation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"

namespace pa {

// Launch with programmatic dependent launch: the grid may start while the
// stream's previous kernel is finishing.  Every partition kernel executes
// griddepcontrol.wait before it touches global memory, so only its launch
// and set-up overlap the previous kernel.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Static facts about one tensor-core partition kernel instantiation.
struct MmaKernelInfo {
  int stage_keys;   // keys per pipeline stage
  int smem_bytes;   // dynamic shared memory
  int ctas_per_sm;  // resident CTAs per SM the launch bounds allow
};

// Per head dim: info and launch of pa_partition_mma<D, kv, nt>.  kv is a
// KvKind, nt the number of 8-row n-tiles per consumer warp.  Return false in
// *ok if the combination is not instantiated.
MmaKernelInfo mma_info_d64(int kv, int nt, bool* ok);
MmaKernelInfo mma_info_d128(int kv, int nt, bool* ok);
MmaKernelInfo mma_info_d256(int kv, int nt, bool* ok);
cudaError_t launch_mma_d64(int kv, int nt, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                           cudaStream_t st);
cudaError_t launch_mma_d128(int kv, int nt, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                            cudaStream_t st);
cudaError_t launch_mma_d256(int kv, int nt, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                            cudaStream_t st);
// head_dim 256, 16-bit caches, pages of 1, 2 or 4 tokens (one n-tile per
// warp, 192 threads): each key's K row arrives by a bulk copy of its own, its
// V row by 16-byte cp.async from a second producer warp.
MmaKernelInfo mma_info_d256_gather(int kv, bool* ok);
cudaError_t launch_mma_d256_gather(int kv, const PartArgs& a, dim3 grid, cudaStream_t st);

// Tensor-memory (tcgen05) partition kernels: head_dim 64 / 128 with KV_BF16 /
// KV_F16 caches.
MmaKernelInfo tc_info(int D, int kv, bool* ok);
cudaError_t launch_tc(int D, int kv, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a, dim3 grid,
                      cudaStream_t st);
// Pages smaller than this many tokens take the cp.async-gather producer of
// the 16-bit tensor-memory kernel (launch_tc forwards them; no tensor maps).
constexpr int kGatherBelowPageSize = 8;
cudaError_t launch_tc_gather(int D, int kv, const PartArgs& a, dim3 grid, cudaStream_t st);

// Prefill tiles of a mixed batch (sequences with more than 8 new tokens):
// up to 256 query rows (two 128-row tiles) per CTA, head_dim 64 / 128,
// KV_BF16 / KV_F16 caches; grid (row blocks, Hkv, key pieces), 320 threads.
cudaError_t launch_prefill_tc(int D, int kv, const CUtensorMap& k, const CUtensorMap& v, const PartArgs& a,
                              dim3 grid, cudaStream_t st);
// Merge of the prefill blocks' key pieces (a.num_parts of them, at most 32)
// into the output rows of the prefill sequences; one warp per row.
cudaError_t launch_prefill_combine(int D, const CombineArgs& a, cudaStream_t st);

// u8 caches, head_dim 128, pages of 16 / 32 / 64 tokens, row tiles n = 16 /
// 32: the keys-on-M tensor-memory kernel with converter warps; stage_keys =
// 128.  Only the K cache needs a tensor map (64-byte swizzled records).
MmaKernelInfo u8_info(int n, int ps, bool* ok);
cudaError_t launch_u8(int n, int ps, const CUtensorMap& k, const PartArgs& a, dim3 grid, cudaStream_t st);

}  // namespace pa
