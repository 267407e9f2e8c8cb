// pa_partition_f32.cuh — split-KV partition kernel for fp32 KV caches.
//
// fp32 caches carry no tensor-core-friendly type, and the workload that uses
// them is small, so this path does plain FFMA: one warp per query row, the
// row's query spread over the lanes, one warp-wide dot product per visible
// key, online softmax in the log2 domain.  It writes the same per-token
// partials as the tensor-core path, so the combine kernel is shared.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D>
__global__ void __launch_bounds__(128) pa_partition_f32(const PartArgs a) {
  constexpr int PER = D / 32;
  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  const SeqInfo si = seq_info(a.begins, a.past_lens, b, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, a.role);
  pdl_launch_dependents();
  if (si.err) {
    if (p == 0 && threadIdx.x == 0) atomicOr(a.status, si.err);
    if (p == 0 && si.rows_ok) {
      const int n = si.T * a.G * D;
      for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        store_out(a.out, a.out_dtype, (static_cast<size_t>(si.t0 + r / a.G) * a.Hq + g * a.G + r % a.G) * D + d,
                  0.f);
      }
    }
    return;
  }
  if (si.T <= 0 || p >= si.nparts) return;
  const int kstart = si.kbase + p * a.part_tokens;
  const int kend = min(kstart + a.part_tokens, si.khi + 1);
  const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;

  if (a.trace != nullptr && threadIdx.x == 0) {
    for (int lp = kstart >> a.ps_log2; lp <= (kend - 1) >> a.ps_log2; ++lp) {
      const int id = __ldg(bt + lp);
      atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
    }
  }

  const float* kc = reinterpret_cast<const float*>(a.k_bytes);
  const float* vc = reinterpret_cast<const float*>(a.v_bytes);
  const int R = si.T * a.G;
  for (int r = warp; r < R; r += blockDim.x / 32) {
    const int i = r / a.G;
    const size_t row = static_cast<size_t>(si.t0 + i) * a.Hq + g * a.G + r % a.G;
    float qv[PER], o[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      qv[e] = load_q_elem(a.q, a.q_dtype, row * D + lane + 32 * e);
      o[e] = 0.f;
    }
    const int p_i = si.L + i;
    const int lo = a.window > 0 ? max(0, p_i - a.window + 1) : 0;
    const uint32_t tm = row_new_token_mask(a.tree_mask, si.t0 + i, i);
    const int hi = a.tree_mask != nullptr ? si.L + si.T - 1 : p_i;
    const int k0 = max(kstart, lo), k1 = min(kend - 1, hi);
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    for (int key = k0; key <= k1; ++key) {
      if (key >= si.L && !((tm >> (key - si.L)) & 1u)) continue;  // a new token outside the row's tree path
      const int id = __ldg(bt + (key >> a.ps_log2));
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
        bad = true;
        break;
      }
      const size_t base = ((static_cast<size_t>(id) * a.Hkv + g) * a.ps + (key & (a.ps - 1))) * D;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) dot = fmaf(qv[e], __ldg(kc + base + lane + 32 * e), dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float s = dot * a.scale_log2;
      const float mnew = fmaxf(m, s);
      const float alpha = ex2(m - mnew);
      const float pw = ex2(s - mnew);
      l = l * alpha + pw;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] = fmaf(pw, __ldg(vc + base + lane + 32 * e), o[e] * alpha);
      m = mnew;
    }
    if (bad && lane == 0) atomicOr(a.status, PA_STATUS_BLOCK_ID);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int d = lane + 32 * e;
      if (si.nparts == 1) {
        store_out(a.out, a.out_dtype, row * D + d, (bad || !(l > 0.f)) ? 0.f : o[e] / l);
      } else {
        const size_t pr = prow(row, si, a.Hq) * a.num_parts + p;
        a.po[pr * D + d] = o[e];
        if (d == 0) {
          a.pm[pr] = m;
          a.pl[pr] = bad ? -1.f : l;
        }
      }
    }
  }
}

}  // namespace pa
