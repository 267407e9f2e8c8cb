// pa_combine.cuh — per-token log-sum-exp combine of the split-KV partials.
//
// One CTA per output row (token t, query head h); its warps split the
// partitions and reduce through shared memory.  The partials are indexed
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

constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) pa_combine(const CombineArgs a) {
  constexpr int PER = D / 32;
  __shared__ float s_acc[kCombineWarps][D];
  __shared__ float s_l[kCombineWarps];
  __shared__ float s_m[kCombineWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;  // one output row (token t, query head h) per CTA
  const int t = static_cast<int>(row / a.Hq);
  // sequence of token t: last b with begins[b] <= t
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.begins + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const SeqInfo si = seq_info(a.begins, a.past_lens, lo, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, a.role);
  pdl_wait_primary();
  pdl_launch_dependents();  // the next step's partition kernel may start its launch
  if (si.foreign) return;  // a prefill chunk of a mixed call: the prefill kernel writes it
  if (si.err || si.T <= 0 || t < si.t0 || t >= si.t0 + si.T) {
    // malformed metadata: the partition kernel reported it; leave zeros
    for (int d = threadIdx.x; d < D; d += blockDim.x) store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + d, 0.f);
    return;
  }
  const int np = si.nparts;
  if (np <= 1) return;  // written directly by the partition kernel
  const size_t pr = prow(static_cast<size_t>(row), si, a.Hq);
  const float* pm = a.pm + pr * a.num_parts;
  const float* pl = a.pl + pr * a.num_parts;
  const float* po = a.po + pr * a.num_parts * D + lane * PER;
  // Warp w merges partitions w, w + 8, ... with its own running max; the
  // loads of up to kBatch partitions are issued together (one round trip).
  constexpr int kBatch = 8;
  float Mw = -INFINITY, lw = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  bool poisoned = false;
  for (int q0 = warp; q0 < np; q0 += kCombineWarps * kBatch) {
    float mq[kBatch], lq[kBatch];
    float x[kBatch][PER];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int q = q0 + kCombineWarps * j;
      const bool ok = q < np;
      mq[j] = ok ? pm[q] : -INFINITY;
      lq[j] = ok ? pl[q] : 0.f;
      const float* src = po + static_cast<size_t>(q) * D;
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const float2 v = ok ? *reinterpret_cast<const float2*>(src + e) : make_float2(0.f, 0.f);
        x[j][e] = v.x;
        x[j][e + 1] = v.y;
      }
    }
    float mnew = Mw;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      mnew = fmaxf(mnew, mq[j]);
      poisoned |= lq[j] < 0.f;
    }
    const float mu = (mnew == -INFINITY) ? 0.f : mnew;
    const float alpha = ex2(Mw - mu);
    lw *= alpha;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= alpha;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = ex2(mq[j] - mu);
      lw += w * lq[j];
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += w * x[j][e];
    }
    Mw = mnew;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
  if (lane == 0) {
    s_l[warp] = lw;
    s_m[warp] = Mw;
  }
  if (__syncthreads_or(poisoned)) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + d, 0.f);
    return;
  }
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, s_m[w]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float wgt[kCombineWarps];
  float lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    wgt[w] = ex2(s_m[w] - Mu);
    lsum += wgt[w] * s_l[w];
  }
  const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) v += wgt[w] * s_acc[w][d];
    store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + d, v * inv);
  }
}

}  // namespace pa
