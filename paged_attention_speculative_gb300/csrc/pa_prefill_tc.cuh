// pa_prefill_tc.cuh — prefill chunks of a mixed batch on the 5th-generation
// tensor cores: sequences with more than 8 new tokens (a chunk of a prompt
// beside the verify steps of other sequences, the MIXED stage of the OpenVINO
// paged-attention op that issue 38153 describes).
//
// One CTA per (row tile, KV head).  A row tile is 128 query rows: TQ = 128 / G
// consecutive new tokens of one sequence times the G query heads of the KV
// head, ordered like the verify kernels' rows (r -> token r / G, head
// g * G + r % G).  The tile streams its keys [klo, khi] once, klo the window
// start of its first token and khi = past_len + its last token, through the
// same pipeline as pa_partition_tc, with every MMA row real:
//   S(s)  = Q . K_s^T   tcgen05.mma M=128, N=64, K=D   (Q in TMEM, K from smem)
//   P(s)  = 2^(S*scale*log2e - m) per row, causal / window mask per row
//   O    += P(s) . V_s  tcgen05.mma M=128, N=D, K=64   (P in TMEM, V from smem)
// and writes the normalised rows directly (no split over keys).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r; warp w reads
//              the lane quarter w)
//   warp 4     MMA issuer (one thread)
//   warp 5     TMA producer: block ids one stage ahead, one tile load per
//              page segment and 128-byte chunk
// Tiles are numbered over the batch's prefill sequences in order, each
// sequence's tiles last token first; each CTA finds its (sequence, first
// token) by walking subsequence_begins.
#pragma once

#include "pa_partition_tc.cuh"

namespace pa {

template <int D, int KV>
__global__ void __launch_bounds__(192, 1)
    pa_prefill_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const PartArgs a) {
  using C = TcCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;                 // [NS] TMA landed
  uint64_t* empty = full + C::NS;        // [NS] stage consumed (MMA commit after PV)
  uint64_t* s_full = empty + C::NS;      // [2] S buffer written (MMA commit)
  uint64_t* s_free = s_full + 2;         // [2] S buffer read (4 softmax warps)
  uint64_t* p_full = s_free + 2;         // [2] P buffer written (4 softmax warps)
  uint64_t* pv_done = p_full + 2;        // [2] PV of the stage using that P buffer done (MMA commit)
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int TQ = 128 / a.G;  // new tokens per row tile
  pdl_wait_primary();        // inputs and outputs may belong to the previous kernel

  // ---- which sequence and tokens this tile covers ----
  int b = -1, i0 = 0;
  {
    long long tile = blockIdx.x;
    for (int s = 0; s < a.num_seqs; ++s) {
      const int T = ld_once(a.begins + s + 1) - ld_once(a.begins + s);
      if (T <= PA_MAX_QUERY_LEN) continue;  // a verify step (or malformed: reported below)
      const long long nt = (T + TQ - 1) / TQ;
      if (tile < nt) {
        // a chunk's tiles in reverse: the last tokens see the most keys, so
        // the longest tiles are scheduled first
        b = s;
        i0 = static_cast<int>(nt - 1 - tile) * TQ;
        break;
      }
      tile -= nt;
    }
  }
  pdl_launch_dependents();
  if (b < 0) return;
  const SeqInfo si = seq_info(a.begins, a.past_lens, b, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, kRoleLong);
  const int nt = min(TQ, si.T - i0);  // tokens of this tile
  const int R = nt * a.G;             // real rows
  if (si.err) {
    if (threadIdx.x == 0) atomicOr(a.status, si.err);
    if (si.rows_ok)
      for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        store_out(a.out, a.out_dtype, (static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G) * D + d,
                  0.f);
      }
    return;
  }
  if (nt <= 0) return;

  const int klo = a.window > 0 ? max(0, si.L + i0 - a.window + 1) : 0;
  const int khi = si.L + i0 + nt - 1;
  const int kstart = (klo >> a.ps_log2) << a.ps_log2;  // page aligned
  const int kend = khi + 1;
  const int n_stages = (kend - kstart + C::SK - 1) / C::SK;

  if (threadIdx.x == 160) {
    s_bad = 0;
    s_timeout = 0;
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t tmem = 0;
  if (warp < 5) {
    if (warp == 0) {
      tmem_alloc(&s_tmem, C::TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
    bar_sync_n(2, 160);  // the TMEM address is published
    tc_fence_after();
    tmem = s_tmem;
    if (warp < 4) {
      // Q rows into TMEM lanes 0..127 (two 16-bit elements per column);
      // rows past the tile's tokens are zero
      const int r = warp * 32 + lane;
      const bool real = r < R;
      const size_t row = real ? static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + row * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = real ? __ldg(src + 8 * c + u) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * u] = x.x;
          v[4 * u + 1] = x.y;
          v[4 * u + 2] = x.z;
          v[4 * u + 3] = x.w;
        }
        tmem_st32(tmem + C::Q_COL + 32 * c + (static_cast<uint32_t>(warp * 32) << 16),
                  reinterpret_cast<const float*>(v));
      }
    }
    tc_fence_before();
    bar_sync_n(2, 160);  // Q is in place for the MMA warp
    tc_fence_after();
  }
  const uint32_t tm_o = tmem;
  const uint32_t tm_s0 = tmem + C::S_COL;
  const uint32_t tm_p0 = tmem + C::P_COL;
  const uint32_t tm_q = tmem + C::Q_COL;

  if (warp == 5) {
    // =========================== TMA producer ===============================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
    const int br_log2 = a.box_log2, br = 1 << br_log2;  // rows per tile load (page size, at most 64)
    int bad = 0;
    // block id of segment `lane` of stage s (0 past the tile's keys)
    auto load_id = [&](int s) -> int {
      const int key = kstart + s * C::SK + (lane << br_log2);
      return (lane < (C::SK >> br_log2) && key < kend) ? __ldg(bt + (key >> a.ps_log2)) : 0;
    };
    int nid = load_id(0);
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % C::NS;
      if (s >= C::NS && !mbar_wait(&empty[slot], ((s / C::NS) - 1) & 1)) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        break;
      }
      int id = nid;
      if (s + 1 < n_stages) nid = load_id(s + 1);
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
        bad = 1;
        id = 0;
      }
      const int key0 = kstart + s * C::SK;
      const int nk = min(C::SK, kend - key0);
      const int nseg = (nk + br - 1) >> br_log2;
      uint8_t* st = smem + slot * C::STAGE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nseg * br * D * 2 * 2));
      __syncwarp();
      const int j = lane;  // one (segment, chunk) pair per lane: nseg * CH <= 16
      const int seg = j / C::CH, c = j % C::CH;
      const int sid = __shfl_sync(0xffffffffu, id, seg & 31);
      if (j < nseg * C::CH) {
        const int key = key0 + (seg << br_log2);
        const uint32_t off = static_cast<uint32_t>((c * C::SK + (seg << br_log2)) * 128);
        tma_load_4d(st + off, &tmK, c * 64, key & (a.ps - 1), g, sid, &full[slot]);
        tma_load_4d(st + C::TILE + off, &tmV, c * 64, key & (a.ps - 1), g, sid, &full[slot]);
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      s_bad = 1;
      atomicOr(a.status, PA_STATUS_BLOCK_ID);
    }
  } else if (warp == 4) {
    // =========================== MMA issuer =================================
    if (lane == 0) {
      bool ok = true;
      auto issue_pv = [&](int s) -> bool {
        const int slot = s % C::NS, pb = s & 1;
        if (!mbar_wait(&p_full[pb], (s >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(smem + slot * C::STAGE + C::TILE);
#pragma unroll
        for (int j = 0; j < C::SK / 16; ++j) {
          const uint64_t bd = sw128_desc(v_base + j * 16 * 128, C::SK * 128, 1024);
          tc_mma_ta(tm_o, tm_p0 + pb * (C::SK / 2) + 8 * j, bd, C::IDESC_PV, (s > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[pb]);
        tc_commit(&empty[slot]);
        return true;
      };
      for (int s = 0; s < n_stages && ok; ++s) {
        const int slot = s % C::NS, sb = s & 1;
        if (!mbar_wait(&full[slot], (s / C::NS) & 1)) {
          ok = false;
          break;
        }
        if (s >= 2 && !mbar_wait(&s_free[sb], ((s >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(smem + slot * C::STAGE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk >> 2, w = kk & 3;
          const uint64_t bd = sw128_desc(k_base + c * C::SK * 128 + 32 * w, 16, 1024);
          tc_mma_ta(tm_s0 + sb * C::SK, tm_q + 8 * kk, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        if (s >= 1) ok = issue_pv(s - 1);
      }
      if (ok && n_stages >= 1) ok = issue_pv(n_stages - 1);
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else {
    // =========================== softmax warps (rows) =======================
    const int r = warp * 32 + lane;  // TMEM lane / query row
    const int rc = min(r, R - 1);    // padding rows mask like the last real row
    const int i = i0 + rc / a.G;     // the row's new token
    const int hi = si.L + i;
    const int lo = a.window > 0 ? si.L + i - a.window + 1 : INT_MIN;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      const int sb = s & 1;
      if (!mbar_wait(&s_full[sb], (s >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[C::SK];
      tmem_ld32(tm_s0 + sb * C::SK + lane_off, x);
      tmem_ld32(tm_s0 + sb * C::SK + 32 + lane_off, x + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);

      const int key0 = kstart + s * C::SK;
      const bool clean = key0 >= lo && key0 + C::SK - 1 <= hi;
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < C::SK; ++j) {
        float v = x[j] * sl2;
        if (!clean) {
          const int key = key0 + j;
          v = (key >= lo && key <= hi) ? v : -INFINITY;
        }
        x[j] = v;
        mt = fmaxf(mt, v);
      }
      const bool need = (mt > m_ref + 8.f) || (m_ref == -INFINITY && mt != -INFINITY);
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? ex2(m_ref - m_new) : 1.f;
      if (__any_sync(0xffffffffu, need) && s >= 1) {
        if (!mbar_wait(&pv_done[(s - 1) & 1], ((s - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tm_o + 32 * c + lane_off, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tm_o + 32 * c + lane_off, o);
        }
        tc_fence_before();
      }
      l *= alpha;
      m_ref = m_new;
      const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[C::SK / 2];
#pragma unroll
      for (int j = 0; j < C::SK; j += 2) {
        const float p0 = ex2(x[j] - mu), p1 = ex2(x[j + 1] - mu);
        l += p0 + p1;
        pk[j / 2] = pack2<C::kBf16>(p0, p1);
      }
      if (s >= 2 && !mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      tmem_st32(tm_p0 + sb * (C::SK / 2) + lane_off, reinterpret_cast<const float*>(pk));
      // V rows of keys outside the tile's range may hold garbage (even NaN):
      // their weights are 0 but 0 * NaN is not, so clear them
      if (key0 < klo || key0 + C::SK - 1 > khi) {
        uint8_t* vt = smem + (s % C::NS) * C::STAGE + C::TILE;
        for (int idx = threadIdx.x; idx < C::SK * C::CH * 8; idx += 128) {
          const int k = idx / (C::CH * 8), rem = idx % (C::CH * 8);
          const int key = key0 + k;
          if (key < klo || key > khi)
            *reinterpret_cast<uint4*>(vt + ((rem >> 3) * C::SK + k) * 128 + 16 * (rem & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    // ---- epilogue: normalised O row from TMEM -> output ----
    if (ok && n_stages >= 1 && !mbar_wait(&pv_done[(n_stages - 1) & 1], ((n_stages - 1) >> 1) & 1)) ok = false;
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
    tc_fence_after();
    const bool poisoned = s_bad != 0 || s_timeout != 0 || !ok;
    const bool real = r < R;
    const size_t row = real ? static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
    const float inv = (poisoned || !(l > 0.f)) ? 0.f : 1.f / l;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32(tm_o + 32 * c + lane_off, o);
      if (real) {
#pragma unroll
        for (int e = 0; e < 32; ++e) store_out(a.out, a.out_dtype, row * D + 32 * c + e, o[e] * inv);
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace pa
