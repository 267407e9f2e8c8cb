// pa_partition_tcu8.cuh — tensor-memory (tcgen05) partition kernel for u8 KV
// caches with per-token fp16 scale / zero-point (OpenVINO issue 38153,
// reproduction step 1: u8 KV cache precision), head_dim 128.
//
// Converter warps dequantise every landed u8 stage once, value by value, to
// f16 ((code - zp) * scale, two f16 operations per pair of codes) in the
// 128-byte-swizzled tile layout of the 16-bit path; from there on the stage
// is processed exactly like an f16 cache (S = Q.K^T and O += P.V on the tensor
// cores, softmax one row per thread).  Keeping the per-key scale and
// zero-point out of the softmax matters: read there, every key costs two
// dependent shared-memory loads on the softmax's critical path.
// Warp roles (256 threads):
//   warps 0, 1    softmax: thread r owns query row r (TMEM lane r)
//   warp 2        MMA issuer (one thread)
//   warp 3        TMA producer: u8 code tiles + per-page scale / zero-point
//   warps 6, 7    converters: u8 stage -> f16 K / V tiles (value rows of keys
//                 outside every query row's range are zeroed: their scales
//                 may be garbage, and 0 * NaN is not 0)
//   warps 4, 5    idle (they wait at the final barrier): warp w issues on
//                 scheduler w % 4, and converters polling next to the
//                 softmax warps would take the issue slots of the softmax
// Rings: u8 stages (TMA -> converters) and f16 buffers (converters -> MMA),
// each released as soon as its consumer is done.
#pragma once

#include "pa_partition_tc.cuh"

namespace pa {

template <int D>
struct TcU8Cfg {
  static_assert(D == 128, "u8 tensor-memory path: head_dim 128");
  static constexpr int ROWS = 64;
  static constexpr int M = 128;
  static constexpr int SK = 64;                           // keys per stage
  static constexpr int CH = D / 64;                       // 128-byte chunks of an f16 key row
  static constexpr int U8_TILE = SK * D;                  // u8 codes of K (or V), [key][128 B]
  static constexpr int U8_SIDE = 8 * SK;                  // [seg][scale|zp] for K, then V
  static constexpr int U8_STAGE = (2 * U8_TILE + U8_SIDE + 1023) / 1024 * 1024;
  static constexpr int F_TILE = SK * D * 2;               // f16 codes of K (or V), [chunk][key][128 B]
  static constexpr int F_STAGE = 2 * F_TILE;
  static constexpr int NB = 3;                            // f16 buffers
  static constexpr int FIXED = NB * F_STAGE + 4 * kMaxPagesPerCta + 512 + 1024;
  static constexpr int NSU_FIT = (226 * 1024 - FIXED) / U8_STAGE;
  static constexpr int NSU = NSU_FIT > 12 ? 12 : NSU_FIT;  // u8 stages
  static constexpr int F_OFF = NSU * U8_STAGE;
  static constexpr int BLK_OFF = F_OFF + NB * F_STAGE;
  static constexpr int BAR_OFF = BLK_OFF + 4 * kMaxPagesPerCta;
  static constexpr int BYTES = BAR_OFF + 512 + 1024;
  static constexpr int S_COL = D;
  static constexpr int P_COL = D + 2 * SK;
  static constexpr int Q_COL = D + 3 * SK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = tc_idesc(M, SK, false, false);
  static constexpr uint32_t IDESC_PV = tc_idesc(M, D, false, true);
  static_assert(NSU >= 3, "u8 ring needs a few stages");
};

template <int D>
__global__ void __launch_bounds__(256, 1)
    pa_partition_tcu8(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const PartArgs a) {
  using C = TcU8Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* fbuf = smem + C::F_OFF;
  int32_t* blk = reinterpret_cast<int32_t*>(smem + C::BLK_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;                // [NSU] u8 stage landed (TMA)
  uint64_t* empty = full + C::NSU;      // [NSU] u8 stage converted (2 converter warps)
  uint64_t* cfull = empty + C::NSU;     // [NB] f16 buffer written (2 converter warps)
  uint64_t* cfree = cfull + C::NB;      // [NB] f16 buffer consumed (MMA commit after PV)
  uint64_t* s_full = cfree + C::NB;     // [2]
  uint64_t* s_free = s_full + 2;        // [2] (2 softmax warps)
  uint64_t* p_full = s_free + 2;        // [2] (2 softmax warps)
  uint64_t* pv_done = p_full + 2;       // [2]
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

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
  const int lp0 = kstart >> a.ps_log2;
  const int npages = ((kend - 1) >> a.ps_log2) - lp0 + 1;
  const int n_stages = (kend - kstart + C::SK - 1) / C::SK;
  const int R = si.T * a.G;

  if (threadIdx.x == 0) {
    s_bad = 0;
    s_timeout = 0;
    for (int s = 0; s < C::NSU; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
    }
    for (int i = 0; i < C::NB; ++i) {
      mbar_init(&cfull[i], 2);
      mbar_init(&cfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 2);
      mbar_init(&p_full[i], 2);
      mbar_init(&pv_done[i], 1);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tm_o = tmem, tm_s0 = tmem + C::S_COL, tm_p0 = tmem + C::P_COL, tm_q = tmem + C::Q_COL;

  // Q rows -> f16 in TMEM (lanes 0..63; softmax warps), zeros in lanes 64..127
  // (warps 2, 3).
  if (warp < 4) {
    const int r = warp * 32 + lane;
    const bool real = r < R;
    const size_t row = real ? static_cast<size_t>(si.t0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + row * D);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t v[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 x = real ? __ldg(src + 8 * c + u) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f;
          if (a.q_dtype == PA_BF16) {
            f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
          } else {
            f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          }
          const __half2 h = __floats2half2_rn(f.x, f.y);
          v[4 * u + e] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      tmem_st32(tm_q + 32 * c + (static_cast<uint32_t>(warp * 32) << 16), reinterpret_cast<const float*>(v));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 3) {
    // =========================== TMA producer ===============================
    int bad = 0;
    for (int j = lane; j < npages; j += 32) {
      int id = __ldg(a.block_tables + static_cast<size_t>(b) * a.max_blocks + lp0 + j);
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
        bad = 1;
        id = 0;
      }
      blk[j] = id;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      s_bad = 1;
      atomicOr(a.status, PA_STATUS_BLOCK_ID);
    }
    __syncwarp();
    const int br_log2 = a.box_log2, br = 1 << br_log2;
    const size_t rec = static_cast<size_t>(a.ps) * (D + 4);
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % C::NSU;
      if (s >= C::NSU && !mbar_wait(&empty[slot], ((s / C::NSU) - 1) & 1)) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        break;
      }
      const int key0 = kstart + s * C::SK;
      const int nk = min(C::SK, kend - key0);
      const int nseg = (nk + br - 1) >> br_log2;
      uint8_t* st = smem + slot * C::U8_STAGE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nseg * br * (2 * D + 8)));
      __syncwarp();
      for (int j = lane; j < nseg; j += 32) {
        const int key = key0 + (j << br_log2);
        const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
        const int id = blk[lp - lp0];
        const uint32_t off = static_cast<uint32_t>((j << br_log2) * 128);
        tma_load_4d(st + off, &tmK, 0, slot0, g, id, &full[slot]);
        tma_load_4d(st + C::U8_TILE + off, &tmV, 0, slot0, g, id, &full[slot]);
        const size_t roff = (static_cast<size_t>(id) * a.Hkv + g) * rec + static_cast<size_t>(a.ps) * D;
        uint8_t* dk = st + 2 * C::U8_TILE + j * 4 * br;
        uint8_t* dv = dk + 4 * C::SK;
        if (br == a.ps) {
          bulk_load(dk, a.k_bytes + roff, 4 * br, &full[slot]);
          bulk_load(dv, a.v_bytes + roff, 4 * br, &full[slot]);
        } else {
          bulk_load(dk, a.k_bytes + roff + 2 * slot0, 2 * br, &full[slot]);
          bulk_load(dk + 2 * br, a.k_bytes + roff + 2 * a.ps + 2 * slot0, 2 * br, &full[slot]);
          bulk_load(dv, a.v_bytes + roff + 2 * slot0, 2 * br, &full[slot]);
          bulk_load(dv + 2 * br, a.v_bytes + roff + 2 * a.ps + 2 * slot0, 2 * br, &full[slot]);
        }
        if (a.trace != nullptr && slot0 == 0)
          atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
      }
    }
  } else if (warp >= 6) {
    // =========================== converters =================================
    const int ct = threadIdx.x - 192;  // 0..63
    const int br_log2 = a.box_log2, br = 1 << br_log2;
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % C::NSU, cb = s % C::NB;
      if (!mbar_wait(&full[slot], (s / C::NSU) & 1)) break;
      if (s >= C::NB && !mbar_wait(&cfree[cb], ((s / C::NB) - 1) & 1)) break;
      const uint8_t* st = smem + slot * C::U8_STAGE;
      uint8_t* fb = fbuf + cb * C::F_STAGE;
      const int key0 = kstart + s * C::SK;
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // K, then V
        const uint8_t* src = st + half * C::U8_TILE;
        const __half* side = reinterpret_cast<const __half*>(st + 2 * C::U8_TILE + half * 4 * C::SK);
        uint8_t* dst = fb + half * C::F_TILE;
#pragma unroll 4
        for (int i = 0; i < (C::SK * 8) / 64; ++i) {
          const int u = ct + 64 * i;                // 16-byte unit of codes
          const int key = u >> 3, us = u & 7;       // d = 16 us .. 16 us + 15
          const int seg = key >> br_log2, o = key & (br - 1);
          const __half sc = side[seg * 2 * br + o], zp = side[seg * 2 * br + br + o];
          // value = code * scale - zp * scale in one rounding; code enters f16
          // exactly (1024 + code, less 1024).  zp * scale is about the size of
          // the values themselves, so its f16 rounding stays relative.
          const __half2 sc2 = __half2half2(sc);
          const __half2 nzs2 = __half2half2(__float2half_rn(-__half2float(zp) * __half2float(sc)));
          const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));
          const bool keep = half == 0 || (key0 + key >= si.klo && key0 + key <= si.khi);
          const uint4 w = *reinterpret_cast<const uint4*>(src + key * 128 + swz(us, key));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
          uint32_t h[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t b = __byte_perm(ws[e], 0x64646464u, q ? 0x4342u : 0x4140u);
              const __half2 v = __hfma2(__hsub2(*reinterpret_cast<__half2*>(&b), k1024), sc2, nzs2);
              h[2 * e + q] = keep ? *reinterpret_cast<const uint32_t*>(&v) : 0u;
            }
          }
          const int c = us >> 2, du = 2 * (us & 3);
          uint8_t* rowp = dst + (c * C::SK + key) * 128;
          *reinterpret_cast<uint4*>(rowp + swz(du, key)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(rowp + swz(du + 1, key)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
      fence_proxy_async();  // f16 tiles are read by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&cfull[cb]);
        mbar_arrive(&empty[slot]);
      }
    }
  } else if (warp >= 4) {
    // idle warps (see the role list above)
  } else if (warp == 2) {
    // =========================== MMA issuer =================================
    if (lane == 0) {
      bool ok = true;
      auto issue_pv = [&](int s) -> bool {
        const int pb = s & 1, cb = s % C::NB;
        if (!mbar_wait(&p_full[pb], (s >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(fbuf + cb * C::F_STAGE + C::F_TILE);
#pragma unroll
        for (int j = 0; j < C::SK / 16; ++j) {
          const uint64_t bd = sw128_desc(v_base + j * 16 * 128, C::SK * 128, 1024);
          tc_mma_ta(tm_o, tm_p0 + pb * (C::SK / 2) + 8 * j, bd, C::IDESC_PV, (s > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[pb]);
        tc_commit(&cfree[cb]);
        return true;
      };
      for (int s = 0; s < n_stages && ok; ++s) {
        const int cb = s % C::NB, sb = s & 1;
        if (!mbar_wait(&cfull[cb], (s / C::NB) & 1)) {
          ok = false;
          break;
        }
        if (s >= 2 && !mbar_wait(&s_free[sb], ((s >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(fbuf + cb * C::F_STAGE);
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
    const int r = warp * 32 + lane;
    const int rc = min(r, R - 1);
    const int hi = si.L + rc / a.G;
    const int lo = a.window > 0 ? hi - a.window + 1 : INT_MIN;
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
        pk[j / 2] = pack2<false>(p0, p1);
      }
      if (s >= 2 && !mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      tmem_st32(tm_p0 + sb * (C::SK / 2) + lane_off, reinterpret_cast<const float*>(pk));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok && n_stages >= 1 && !mbar_wait(&pv_done[(n_stages - 1) & 1], ((n_stages - 1) >> 1) & 1)) ok = false;
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
    tc_fence_after();
    const bool poisoned = s_bad != 0 || s_timeout != 0 || !__all_sync(0xffffffffu, ok);
    const bool real = r < R;
    const size_t row = real ? static_cast<size_t>(si.t0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      tmem_ld32(tm_o + 32 * c + lane_off, o);
      if (real) {
        if (si.nparts == 1) {
          const float inv = (poisoned || !(l > 0.f)) ? 0.f : 1.f / l;
#pragma unroll
          for (int e = 0; e < 32; ++e) store_out(a.out, a.out_dtype, row * D + 32 * c + e, o[e] * inv);
        } else {
          float4* dst = reinterpret_cast<float4*>(a.po + (prow(row, si, a.Hq) * a.num_parts + p) * D + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
      }
    }
    if (real && si.nparts > 1) {
      a.pm[prow(row, si, a.Hq) * a.num_parts + p] = m_ref;
      a.pl[prow(row, si, a.Hq) * a.num_parts + p] = poisoned ? -1.f : l;
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
