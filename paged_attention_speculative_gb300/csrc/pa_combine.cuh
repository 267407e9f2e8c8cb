// pa_combine.cuh — per-token log-sum-exp combine of the split-KV partials.
//
// Two output rows (token t, query head h) per CTA; four warps per row split
// its partitions and reduce through shared memory.  The partials are indexed
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
constexpr int kCombineRows = 2;                              // output rows per CTA
constexpr int kWarpsPerRow = kCombineWarps / kCombineRows;  // warps splitting one row's partitions

// Two rows per CTA, four warps per row: half as many CTAs as rows, so that
// more of them are resident (waiting in griddepcontrol.wait) before the
// partition grid ends -- a CTA that only starts once it ends pays its index
// work and metadata loads on the critical path.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32, 4) pa_combine(const CombineArgs a) {
  constexpr int PER = D / 32;
  __shared__ float s_acc[kCombineWarps][D];
  __shared__ float s_l[kCombineWarps];
  __shared__ float s_m[kCombineWarps];
  __shared__ int s_bad[kCombineRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = warp / kWarpsPerRow, wq = warp % kWarpsPerRow;  // row of the CTA, warp within the row
  const long long rows = static_cast<long long>(a.total_tokens) * a.Hq;
  const long long row = static_cast<long long>(blockIdx.x) * kCombineRows + sub;
  const bool live = row < rows;
  const int t = live ? static_cast<int>(row / a.Hq) : 0;
  // sequence of token t: last b with begins[b] <= t
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.begins + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const SeqInfo si = seq_info(a.begins, a.past_lens, lo, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, a.role);
  if (threadIdx.x < kCombineRows) s_bad[threadIdx.x] = 0;
  __syncthreads();  // the flags are clear before any warp can raise one
  pdl_wait_primary();
  pdl_launch_dependents();  // the next step's partition kernel may start its launch
  // what this row needs: 0 nothing (another kernel writes it), 1 zeros
  // (malformed metadata, reported by the partition kernel), 2 the merge
  int mode = 2;
  if (!live || si.foreign) mode = 0;
  else if (si.err || si.T <= 0 || t < si.t0 || t >= si.t0 + si.T) mode = 1;
  else if (si.nparts <= 1) mode = 0;  // written directly by the partition kernel
  const int np = si.nparts;
  float Mw = -INFINITY, lw = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  bool poisoned = false;
  if (mode == 2) {
    const size_t pr = prow(static_cast<size_t>(row), si, a.Hq);
    const float* pm = a.pm + pr * a.num_parts;
    const float* pl = a.pl + pr * a.num_parts;
    const float* po = a.po + pr * a.num_parts * D + lane * PER;
    // Warp wq merges partitions wq, wq + 4, ... with its own running max; the
    // loads of up to kBatch partitions are issued together (one round trip).
    constexpr int kBatch = 5;  // 4 warps x 5: up to 20 partitions per round trip
    for (int q0 = wq; q0 < np; q0 += kWarpsPerRow * kBatch) {
      float mq[kBatch], lq[kBatch];
      float x[kBatch][PER];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int q = q0 + kWarpsPerRow * j;
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
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
  if (lane == 0) {
    s_l[warp] = lw;
    s_m[warp] = Mw;
  }
  if (poisoned) s_bad[sub] = 1;
  __syncthreads();
  if (mode == 0) return;
  const int w0 = sub * kWarpsPerRow;
  const bool zero = mode == 1 || s_bad[sub] != 0;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarpsPerRow; ++w) M = fmaxf(M, s_m[w0 + w]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float wgt[kWarpsPerRow];
  float lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kWarpsPerRow; ++w) {
    wgt[w] = ex2(s_m[w0 + w] - Mu);
    lsum += wgt[w] * s_l[w0 + w];
  }
  const float inv = (zero || !(lsum > 0.f)) ? 0.f : 1.f / lsum;
  // this row's kWarpsPerRow warps write its D outputs, four per thread
  for (int d = 4 * (wq * 32 + lane); d < D; d += 4 * 32 * kWarpsPerRow) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarpsPerRow; ++w) {
      v.x += wgt[w] * s_acc[w0 + w][d];
      v.y += wgt[w] * s_acc[w0 + w][d + 1];
      v.z += wgt[w] * s_acc[w0 + w][d + 2];
      v.w += wgt[w] * s_acc[w0 + w][d + 3];
    }
    store_out4(a.out, a.out_dtype, static_cast<size_t>(row) * D + d,
               make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv));
  }
}

}  // namespace pa
