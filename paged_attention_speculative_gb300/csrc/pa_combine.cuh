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
               zero ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv));
  }
}

}  // namespace pa

namespace pa {

// Prefill chunks whose blocks' keys were split into S pieces (S <=
// a.num_parts, the partial rows' stride; the same count the prefill kernel
// derives from the batch): one warp per output row (token t, query head h)
// of a prefill sequence merges the row's S partials [t * Hq + h][piece] with
// the same log-sum-exp rule.  Rows of verify steps (T_b <= 8) and of sequences with malformed
// metadata (which the prefill kernel zeroed and reported) are left alone.
template <int D>
__global__ void __launch_bounds__(128) pa_prefill_combine(const CombineArgs a) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const long long rows = static_cast<long long>(a.total_tokens) * a.Hq;
  const int t = row < rows ? static_cast<int>(row / a.Hq) : 0;
  int lo = 0, hi = a.num_seqs - 1;  // sequence of token t: last b with begins[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.begins + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const SeqInfo si = seq_info(a.begins, a.past_lens, lo, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, kRoleLong);
  const int S = prefill_pieces(a.begins, a.num_seqs, a.row_cap / a.G, a.Hkv, a.num_parts, a.num_sms);
  pdl_wait_primary();
  pdl_launch_dependents();
  if (S <= 1 || row >= rows || si.foreign || si.err || t < si.t0 || t >= si.t0 + si.T) return;
  // the pieces of this row's block (its TQ tokens and their keys), as the
  // prefill kernel counts them; one piece: the kernel wrote the row itself
  const int TQ = a.row_cap / a.G;
  const int i0 = (t - si.t0) / TQ * TQ, ntok = min(TQ, si.T - i0);
  const int klo = a.window > 0 ? max(0, si.L + i0 - a.window + 1) : 0;
  const int pieces = prefill_block_pieces(S, si.L + i0 + ntok - (klo / a.ps) * a.ps);
  if (pieces <= 1) return;
  const size_t pr = static_cast<size_t>(row) * a.num_parts;  // pieces [0, pieces) of at most 32, one per lane
  const float mj = lane < pieces ? a.pm[pr + lane] : -INFINITY;
  const float lj = lane < pieces ? a.pl[pr + lane] : 0.f;
  float M = mj;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float Mu = (M == -INFINITY) ? 0.f : M;
  const float wj = ex2(mj - Mu);
  float lsum = wj * lj;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
  const bool poisoned = __any_sync(0xffffffffu, lj < 0.f);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  const float* po = a.po + pr * D + lane * PER;
  for (int j = 0; j < pieces; ++j) {
    const float w = __shfl_sync(0xffffffffu, wj, j);
#pragma unroll
    for (int e = 0; e < PER; e += 2) {
      const float2 v = *reinterpret_cast<const float2*>(po + static_cast<size_t>(j) * D + e);
      acc[e] = fmaf(w, v.x, acc[e]);
      acc[e + 1] = fmaf(w, v.y, acc[e + 1]);
    }
  }
  const float inv = (poisoned || !(lsum > 0.f)) ? 0.f : 1.f / lsum;
#pragma unroll
  for (int e = 0; e < PER; ++e) store_out(a.out, a.out_dtype, static_cast<size_t>(row) * D + lane * PER + e,
                                 poisoned ? 0.f : acc[e] * inv);
}

}  // namespace pa
