// pa_combine.cuh — per-token log-sum-exp combine of the split-KV partials.
//
// One warp per output row (token t, query head h).  The partials are indexed
// per query token — [t, h, partition] — so any number of new tokens per
// sequence keeps the split (the per-sequence buffer the dual-radeon-vllm
// article, use_3d section, identifies as the reason the split path was
// disabled for more than one query row).  With partition p holding running
// max m_p (log2 domain), denominator l_p and unnormalised output o_p:
//   M = max_p m_p,  out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p.
// Launched with programmatic dependent launch: index work runs while the
// partition grid drains; griddepcontrol.wait guards the reads of partials.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D>
__global__ void __launch_bounds__(128) pa_combine(const CombineArgs a) {
  constexpr int PER = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (row >= static_cast<long long>(a.total_tokens) * a.Hq) return;
  const int t = static_cast<int>(row / a.Hq);
  // sequence of token t: last b with begins[b] <= t
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.begins + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const SeqInfo si = seq_info(a.begins, a.past_lens, lo, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap);
  pdl_wait_primary();
  if (si.err || si.T <= 0 || t < si.t0 || t >= si.t0 + si.T) {
    // malformed metadata: the partition kernel reported it; leave zeros
    for (int e = 0; e < PER; ++e) store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + lane + 32 * e, 0.f);
    return;
  }
  const int np = si.nparts;
  if (np <= 1) return;  // written directly by the partition kernel
  const float* pm = a.pm + static_cast<size_t>(row) * a.num_parts;
  const float* pl = a.pl + static_cast<size_t>(row) * a.num_parts;
  float M = -INFINITY;
  bool poisoned = false;
  for (int q = lane; q < np; q += 32) {
    M = fmaxf(M, pm[q]);
    poisoned |= pl[q] < 0.f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  poisoned = __any_sync(0xffffffffu, poisoned);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float lsum = 0.f;
  for (int q = lane; q < np; q += 32) lsum += ex2(pm[q] - Mu) * pl[q];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);

  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  const float* po = a.po + static_cast<size_t>(row) * a.num_parts * D;
  for (int q = 0; q < np; ++q) {
    const float w = ex2(pm[q] - Mu);
    const float* src = po + static_cast<size_t>(q) * D + lane * PER;
    if constexpr (PER == 8) {
      const float4 x0 = *reinterpret_cast<const float4*>(src);
      const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
      acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
      acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
    } else if constexpr (PER == 4) {
      const float4 x0 = *reinterpret_cast<const float4*>(src);
      acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
    } else {
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += w * src[e];
    }
  }
  const bool zero = poisoned || !(lsum > 0.f);
  const float inv = zero ? 0.f : 1.f / lsum;
#pragma unroll
  for (int e = 0; e < PER; ++e)
    store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + lane * PER + e, acc[e] * inv);
}

}  // namespace pa
