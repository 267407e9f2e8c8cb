// pa_partition_tku8.cuh — keys-on-M tensor-memory partition kernel for u8 KV
// caches with per-token fp16 scale / zero-point (OpenVINO issue 38153,
// reproduction step 1: u8 KV cache precision), head_dim 128, up to 32 query
// rows per KV head.
//
// With a key per softmax thread the per-key dequantisation terms are scalars
// of that thread, so the tensor cores can run on the raw codes (exact in f16)
// and the terms are applied around them (value = (code - zp) * scale):
//   S^T[k][n]  = ks_k * (C_k . q_n  -  kz_k * sum_d q_n)     C_k = K codes of key k
//   P'[k][n]   = 2^(S^T scale log2e - m_n) * vs_k            (f16, what the MMA reads)
//   O^T[d][n] += sum_k Vc[k][d] P'[k][n]                      Vc = V codes
//   out[n][d]  = (O^T[d][n] - sum_k P'[k][n] vz_k) / sum_k 2^(...)
// The correction sum_k P' vz_k is accumulated from the same rounded P' that the
// MMA multiplies, so the subtraction is exact up to fp32 rounding.
//
// Warp roles (320 threads):
//   warps 0..3  softmax: warp w owns TMEM lanes 32w..32w+31 (keys / head dims)
//   warps 4..7  converters: thread t of warp 4+w (TMEM lane 32w+t) turns the K
//               codes of key 32w+t of a 128-key stage into f16 in TMEM (A
//               operand of S^T), gathers head dim 32w+t of every key's V codes
//               into TMEM (A operand of O^T = V^T P'^T), and writes key 32w+t's
//               scale / zero-point to a side buffer (zero for keys out of range)
//   warp 8      MMA issuer (one thread)
//   warp 9      TMA producer: u8 code tiles + per-page scales / zero-points,
//               in 64-key half stages
#pragma once

#include "pa_partition_tk.cuh"

namespace pa {

template <int N>
struct TkU8Cfg {
  static_assert(N == 16 || N == 32, "row tile 16 / 32");
  static constexpr int D = 128;
  static constexpr int SK = 128;                       // keys per stage (M of the score MMA)
  static constexpr int HK = 64;                        // keys per u8 half stage
  static constexpr int U8_TILE = HK * D;               // u8 codes of K (or V), [key][128 B]
  static constexpr int U8_SIDE = 8 * HK;               // [seg][scale|zp] for K, then V
  static constexpr int U8_STAGE = (2 * U8_TILE + U8_SIDE + 1023) / 1024 * 1024;
  static constexpr int SIDE = SK * 16;                 // float4 per key: ks*scale*log2e, kz, vs, vz
  static constexpr int NB = 3;                         // converted stages in flight
  static constexpr int Q_BYTES = N * D * 2;
  static constexpr int P_BYTES = N * SK * 2;          // P'^T, K-major: [key chunk][row][128 B]
  static constexpr int MISC = 4608;
  static constexpr int FIXED = NB * SIDE + Q_BYTES + 2 * P_BYTES + 4 * kMaxPagesPerCta + MISC + 1024;
  static constexpr int NSU_FIT = (226 * 1024 - FIXED) / U8_STAGE;
  static constexpr int NSU = NSU_FIT > 12 ? 12 : NSU_FIT;  // u8 half stages in the ring
  static constexpr int SIDE_OFF = NSU * U8_STAGE;
  static constexpr int Q_OFF = SIDE_OFF + NB * SIDE;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int BLK_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int MISC_OFF = BLK_OFF + 4 * kMaxPagesPerCta;
  static constexpr int BYTES = MISC_OFF + MISC + 1024;
  // TMEM columns: O^T [0, N), S^T [N, 3N), K codes [K_COL + 64 b, +64),
  // V^T codes [V_COL + 64 b, +64) (two f16 per column)
  static constexpr int K_COL = 3 * N <= 64 ? 64 : 128;
  static constexpr int V_COL = K_COL + 64 * NB;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = tk_idesc(128, N, false, false, false);
  static constexpr uint32_t IDESC_PV = tk_idesc(128, N, false, false, false);
  static_assert(3 * N <= K_COL, "tensor-memory budget");
  static_assert(NSU >= 4, "u8 ring needs a few half stages");
  static_assert(V_COL + 64 * NB <= TMEM_COLS, "tensor-memory budget");
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0, "swizzled tiles are 1024-aligned");
};

template <int N>
__global__ void __launch_bounds__(320, 1)
    pa_partition_tku8(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const PartArgs a) {
  using C = TkU8Cfg<N>;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float4* side_buf = reinterpret_cast<float4*>(smem + C::SIDE_OFF);   // [NB][SK]
  uint8_t* qt = smem + C::Q_OFF;
  uint8_t* pt = smem + C::P_OFF;
  int32_t* blk = reinterpret_cast<int32_t*>(smem + C::BLK_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::MISC_OFF);
  uint64_t* full = bars;                 // [NSU] u8 half stage landed (TMA)
  uint64_t* empty = full + C::NSU;       // [NSU] u8 half stage converted (4 converter warps)
  uint64_t* cfull = empty + C::NSU;      // [NB] stage converted (4 converter warps)
  uint64_t* cfree = cfull + C::NB;       // [NB] converted stage consumed (MMA commit after PV)
  uint64_t* s_full = cfree + C::NB;      // [2]
  uint64_t* s_free = s_full + 2;         // [2] (4 softmax warps)
  uint64_t* p_full = s_free + 2;         // [2] (4 softmax warps)
  uint64_t* pv_done = p_full + 2;        // [2]
  float* m_sm = reinterpret_cast<float*>(smem + C::MISC_OFF + 512);   // [64] row reference maxima
  float* xch = m_sm + 64;                                             // [4][64] per-warp row values
  float* m_next = xch + 256;                                          // [64]
  float* alpha_sm = m_next + 64;                                      // [64]
  long long* rowoff = reinterpret_cast<long long*>(alpha_sm + 64);    // [64]
  float* qsum_sm = reinterpret_cast<float*>(rowoff + 64);             // [64] sum_d of each f16 query row
  float* xch2 = qsum_sm + 64;                                         // [4][64] second exchange
  uint32_t* tree_rows = reinterpret_cast<uint32_t*>(xch2 + 256);      // [8] rows that see new token k
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  const bool prefetch = (warp == 9 && a.window == 0);
  if (prefetch) {
    const long long lpg = (static_cast<long long>(p) * a.part_tokens) >> a.ps_log2;
    const int n = static_cast<int>(min(static_cast<long long>(a.part_tokens >> a.ps_log2),
                                       max(0LL, static_cast<long long>(a.max_blocks) - lpg)));
    const int32_t* src = a.block_tables + static_cast<size_t>(b) * a.max_blocks + lpg;
    for (int j = lane; j < n; j += 32) cp_async4(blk + j, src + j);
  }
  const SeqInfo si = seq_info(a.begins, a.past_lens, b, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, a.role);
  pdl_launch_dependents();
  if (si.err || si.T <= 0 || p >= si.nparts) {
    if (prefetch) cp_async_wait_all();
  }
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
  const float sl2 = a.scale_log2;

  if (threadIdx.x == 288) {
    s_bad = 0;
    s_timeout = 0;
    for (int i = 0; i < C::NSU; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    for (int i = 0; i < C::NB; ++i) {
      mbar_init(&cfull[i], 4);
      mbar_init(&cfree[i], 1);
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
  bool ok = true;
  uint32_t tmem = 0;
  if (warp == 0) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Q rows -> f16, K-major swizzled tile (rows R..N-1 zero); then the sum of
    // each f16 row, in head-dim order
    for (int idx = threadIdx.x; idx < N * (D / 8); idx += 128) {
      const int n = idx / (D / 8), u16 = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < R) {
        const size_t row = static_cast<size_t>(si.t0 + n / a.G) * a.Hq + g * a.G + n % a.G;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + row * D) + u16);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = (a.q_dtype == PA_BF16) ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]))
                                                  : __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          const __half2 hh = __floats2half2_rn(f.x, f.y);
          h[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        v = make_uint4(h[0], h[1], h[2], h[3]);
      }
      *reinterpret_cast<uint4*>(qt + ((u16 >> 3) * N + n) * 128 + swz(u16 & 7, n)) = v;
    }
    if (threadIdx.x < 64) m_sm[threadIdx.x] = -INFINITY;
    fence_proxy_async();  // the Q tile is read by the tensor cores
    bar_sync_n(1, 128);
    if (threadIdx.x < N) {
      const int n = threadIdx.x;
      float sum = 0.f;
      for (int u16 = 0; u16 < D / 8; ++u16) {
        const uint4 x = *reinterpret_cast<const uint4*>(qt + ((u16 >> 3) * N + n) * 128 + swz(u16 & 7, n));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          sum += f.x;
          sum += f.y;
        }
      }
      qsum_sm[n] = sum;
    }
    if (threadIdx.x < PA_MAX_QUERY_LEN) {
      // tree masks: the rows that see new token k (row n = token n / G)
      const int k = threadIdx.x;
      uint32_t rows = 0;
      if (a.tree_mask != nullptr)
        for (int n = 0; n < R; ++n) rows |= ((ld_once_u8(a.tree_mask + si.t0 + n / a.G) >> k) & 1u) << n;
      tree_rows[k] = rows;
    }
  }
  if (warp < 9) {
    // TMEM address, Q tile and row sums published to softmax, converter and MMA warps
    tc_fence_before();
    bar_sync_n(2, 288);
    tc_fence_after();
    tmem = s_tmem;
  }
  const uint32_t tm_o = tmem;            // O^T: lane = head dim, column = row
  const uint32_t tm_s0 = tmem + N;       // S^T buffers: lane = key, column = row
  const uint32_t tm_k = tmem + C::K_COL; // K codes: lane = key, two f16 per column
  const uint32_t tm_v = tmem + C::V_COL; // V^T codes: lane = head dim, two keys per column

  if (warp == 9) {
    // =========================== TMA producer ===============================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    int bad = 0;
    if (prefetch) {
      cp_async_wait_all();
      __syncwarp();
    }
    for (int j = lane; j < npages; j += 32) {
      int id = prefetch ? blk[j] : __ldg(a.block_tables + static_cast<size_t>(b) * a.max_blocks + lp0 + j);
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
    const int halves = 2 * n_stages;
    int issued = 0;
    for (int i = 0; i < halves; ++i, ++issued) {
      const int slot = i % C::NSU;
      if (i >= C::NSU && !mbar_wait(&empty[slot], ((i / C::NSU) - 1) & 1)) {
        ok = false;
        break;
      }
      const int key0 = kstart + i * C::HK;
      const int nk = max(0, min(C::HK, kend - key0));
      const int nseg = (nk + br - 1) >> br_log2;
      uint8_t* st = smem + slot * C::U8_STAGE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nseg * br * (2 * D + 8)));
      __syncwarp();
      // one copy per lane (a copy instruction costs its thread hundreds of
      // cycles): K and V code tiles, then the pages' scales / zero-points
      const bool whole = (br == a.ps);
      const int ncopy = nseg * (whole ? 4 : 6);
      for (int c = lane; c < ncopy; c += 32) {
        if (c < 2 * nseg) {
          const bool is_v = c >= nseg;
          const int j = is_v ? c - nseg : c;
          const int key = key0 + (j << br_log2);
          const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
          const int id = blk[lp - lp0];
          const uint32_t off = static_cast<uint32_t>((j << br_log2) * 128);
          tma_load_4d(st + (is_v ? C::U8_TILE : 0) + off, is_v ? &tmV : &tmK, 0, slot0, g, id, &full[slot]);
          if (!is_v && a.trace != nullptr && slot0 == 0)
            atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
        } else {
          const int idx = c - 2 * nseg;
          const int j = whole ? idx >> 1 : idx >> 2;
          const bool is_v = whole ? (idx & 1) != 0 : (idx & 2) != 0;
          const int part = whole ? 0 : (idx & 1);  // 0: scales, 1: zero-points
          const int key = key0 + (j << br_log2);
          const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
          const int id = blk[lp - lp0];
          const size_t roff = (static_cast<size_t>(id) * a.Hkv + g) * rec + static_cast<size_t>(a.ps) * D;
          uint8_t* dst = st + 2 * C::U8_TILE + j * 4 * br + (is_v ? 4 * C::HK : 0);
          const uint8_t* src = (is_v ? a.v_bytes : a.k_bytes) + roff;
          if (whole) bulk_load(dst, src, 4 * br, &full[slot]);
          else bulk_load(dst + 2 * br * part, src + 2 * a.ps * part + 2 * slot0, 2 * br, &full[slot]);
        }
      }
    }
    if (lane == 0) {
      for (int i = max(0, issued - C::NSU); i < issued; ++i)
        if (!mbar_wait(&full[i % C::NSU], (i / C::NSU) & 1)) ok = false;
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // =========================== converters =================================
    const int ct = threadIdx.x - 128;                         // key of the stage, 0..127
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const int br_log2 = a.box_log2, br = 1 << br_log2;
    for (int s = 0; s < n_stages && ok; ++s) {
      const int cb = s % C::NB, h0 = 2 * s, h1 = 2 * s + 1;
      if (!mbar_wait(&full[h0 % C::NSU], (h0 / C::NSU) & 1) || !mbar_wait(&full[h1 % C::NSU], (h1 / C::NSU) & 1) ||
          (s >= C::NB && !mbar_wait(&cfree[cb], ((s / C::NB) - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // K codes of key ct -> f16 pairs in TMEM (column j holds head dims 2j, 2j+1)
      {
        const int hk = ct >> 6, r = ct & 63;
        const uint8_t* st = smem + ((h0 + hk) % C::NSU) * C::U8_STAGE;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(st + r * 128 + swz(4 * half + u, r));
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              w[8 * u + 2 * e] = u8pair_to_f16x2(xs[e], 0x4140u);
              w[8 * u + 2 * e + 1] = u8pair_to_f16x2(xs[e], 0x4342u);
            }
          }
          tmem_st32(tm_k + cb * 64 + 32 * half + lane_off, reinterpret_cast<const float*>(w));
        }
        // the key's dequantisation terms; zero outside every row's range
        // (there the scales may be garbage)
        const int seg = r >> br_log2, o = r & (br - 1);
        const __half* ks = reinterpret_cast<const __half*>(st + 2 * C::U8_TILE + seg * 4 * br);
        const __half* vs = reinterpret_cast<const __half*>(st + 2 * C::U8_TILE + 4 * C::HK + seg * 4 * br);
        const int key = kstart + s * C::SK + ct;
        const bool in = key >= si.klo && key <= si.khi && key < kend;  // past kend: the next partition's
        side_buf[cb * C::SK + ct] = in ? make_float4(__half2float(ks[o]) * sl2, __half2float(ks[br + o]),
                                                     __half2float(vs[o]), __half2float(vs[br + o]))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // V^T: this thread's head dim dv of every key -> f16 pairs (keys 2j, 2j+1
      // in column j).  The byte of key r (row r of a half stage's swizzled
      // [key][128 B] tile) sits in the 32-bit word at r * 128 +
      // ((dv / 16) ^ (r % 8)) * 16 + (dv % 16 & ~3).
      {
        const int dv = ct;
        const int du = dv >> 4, dsel = dv & 3;
        uint32_t off[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) off[i] = 128 * i + ((du ^ i) << 4) + (dv & 12);
        const uint32_t sel = static_cast<uint32_t>(dsel | ((4 + dsel) << 4));  // bytes: a.dsel, b.dsel
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          const uint8_t* vt = smem + ((h0 + hk) % C::NSU) * C::U8_STAGE + C::U8_TILE;
          uint32_t w[32];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              const uint32_t a0 = *reinterpret_cast<const uint32_t*>(vt + 1024 * m + off[i]);
              const uint32_t a1 = *reinterpret_cast<const uint32_t*>(vt + 1024 * m + off[i + 1]);
              const uint32_t t = __byte_perm(a0, a1, sel);
              w[4 * m + i / 2] = u8pair_to_f16x2(t, 0x4140u);
            }
          }
          tmem_st32(tm_v + cb * 64 + 32 * hk + lane_off, reinterpret_cast<const float*>(w));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&cfull[cb]);
        mbar_arrive(&empty[h0 % C::NSU]);
        mbar_arrive(&empty[h1 % C::NSU]);
      }
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
  } else if (warp == 8) {
    // =========================== MMA issuer =================================
    // Issues S^T(s) as soon as stage s is converted and its S^T buffer is
    // free, and PV(s) as soon as P'(s) is written, whichever comes first.
    if (lane == 0) {
      const uint32_t q_base = smem_u32(qt);
      int ns = 0, np = 0;
      uint32_t idle = 0;
      while (np < n_stages) {
        bool progress = false;
        if (ns < n_stages && mbar_test(&cfull[ns % C::NB], (ns / C::NB) & 1) &&
            (ns < 2 || mbar_test(&s_free[ns & 1], ((ns >> 1) - 1) & 1))) {
          const int cb = ns % C::NB, sb = ns & 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk >> 2, w = kk & 3;
            const uint64_t bd = sw128_desc(q_base + c * N * 128 + 32 * w, 16, 1024);
            tc_mma_ta(tm_s0 + sb * N, tm_k + cb * 64 + 8 * kk, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[sb]);
          ++ns;
          progress = true;
        }
        if (np < ns && mbar_test(&p_full[np & 1], (np >> 1) & 1)) {
          const int pb = np & 1, cb = np % C::NB;
          tc_fence_after();
          const uint32_t p_base = smem_u32(pt + pb * C::P_BYTES);
#pragma unroll
          for (int j = 0; j < C::SK / 16; ++j) {
            const uint64_t bd = sw128_desc(p_base + (j >> 2) * N * 128 + 32 * (j & 3), 16, 1024);
            tc_mma_ta(tm_o, tm_v + cb * 64 + 8 * j, bd, C::IDESC_PV, (np > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit(&pv_done[pb]);
          tc_commit(&cfree[cb]);
          ++np;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else if (++idle > kWaitLimit) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
          break;
        }
      }
    }
    __syncwarp();
  }

  // =========================== softmax warps (keys) ==========================
  float l[N], zc[N];
  if (warp < 4) {
    const int kq = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float qs[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
      l[n] = 0.f;
      zc[n] = 0.f;
      qs[n] = qsum_sm[n];
    }
    for (int s = 0; s < n_stages; ++s) {
      const int sb = s & 1, cb = s % C::NB;
      if (ok) ok = mbar_wait(&s_full[sb], (s >> 1) & 1);
      tc_fence_after();
      float v[N];
      tmem_ld_n<N>(tm_s0 + sb * N + lane_off, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      // this key's dequantisation terms (written by the converters before cfull)
      if (ok) ok = mbar_wait(&cfull[cb], (s / C::NB) & 1);
      const float4 sd = side_buf[cb * C::SK + kq];

      const int key = kstart + s * C::SK + kq;
      const int dk = key - si.L;
      // rows that see this key, as a bit set: [nlo, nhi) (the causal limit
      // and the window), or for a tree mask the window and the rows whose
      // mask names this new token
      const bool tree = a.tree_mask != nullptr;
      const int nlo = (dk > 0 && !tree) ? dk * a.G : 0;
      int nhi = R;
      if (a.window > 0) nhi = min(R, max(0, (dk + a.window) * a.G));
      if (key >= kend) nhi = 0;  // a half-filled last stage: those keys belong to the next partition
      const uint32_t below_hi = nhi >= 32 ? 0xffffffffu : ((1u << nhi) - 1u);
      const uint32_t below_lo = nlo >= 32 ? 0xffffffffu : ((1u << nlo) - 1u);
      uint32_t vrows = below_hi & ~below_lo;
      if (tree && dk >= 0) vrows &= (dk < PA_MAX_QUERY_LEN) ? tree_rows[dk] : 0u;
      const bool clean = (nlo == 0 && nhi >= R) && !(tree && dk >= 0);
      bool need = false;
#pragma unroll
      for (int n4 = 0; n4 < N; n4 += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_sm + n4);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = n4 + e;
          float x = fmaf(-sd.y, qs[n], v[n]) * sd.x;
          if (!clean) x = ((vrows >> n) & 1u) ? x : -INFINITY;
          v[n] = x;
          need |= x > mm[e] + 8.f;
        }
      }
      if (bar_any(1, 128, need)) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
          float t = v[n];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
          if (lane == 0) xch[warp * 64 + n] = t;
        }
        bar_sync_n(1, 128);
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const float rm = fmaxf(fmaxf(xch[n], xch[64 + n]), fmaxf(xch[128 + n], xch[192 + n]));
          const float mo = m_sm[n];
          const float mn = rm > mo + 8.f ? rm : mo;
          const float al = (mn == mo) ? 1.f : ex2(mo - mn);
          l[n] *= al;
          zc[n] *= al;
          if (n == threadIdx.x) {
            m_next[n] = mn;
            alpha_sm[n] = al;
          }
        }
        bar_sync_n(1, 128);
        if (threadIdx.x < N) m_sm[threadIdx.x] = m_next[threadIdx.x];
        if (s >= 1) {
          if (ok) ok = mbar_wait(&pv_done[(s - 1) & 1], ((s - 1) >> 1) & 1);
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < N / 16; ++c) {
            float o[16];
            tmem_ld16(tm_o + 16 * c + lane_off, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha_sm[16 * c + e];
            tmem_st16(tm_o + 16 * c + lane_off, reinterpret_cast<const uint32_t*>(o));
          }
          tc_fence_before();
        }
        bar_sync_n(1, 128);
      }
      // weights times the key's V scale, rounded to f16 as the MMA reads them;
      // the zero-point correction uses the rounded values
      uint32_t pk[N / 2];
#pragma unroll
      for (int n4 = 0; n4 < N; n4 += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_sm + n4);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const float mu0 = mm[e] == -INFINITY ? 0.f : mm[e];
          const float mu1 = mm[e + 1] == -INFINITY ? 0.f : mm[e + 1];
          const float p0 = ex2(v[n4 + e] - mu0), p1 = ex2(v[n4 + e + 1] - mu1);
          l[n4 + e] += p0;
          l[n4 + e + 1] += p1;
          const __half2 h = __floats2half2_rn(p0 * sd.z, p1 * sd.z);
          const float2 hr = __half22float2(h);
          zc[n4 + e] = fmaf(hr.x, sd.w, zc[n4 + e]);
          zc[n4 + e + 1] = fmaf(hr.y, sd.w, zc[n4 + e + 1]);
          pk[(n4 + e) / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      if (s >= 2 && ok) ok = mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1);
      // P'^T, K-major: row n holds the stage's 128 keys (two 128-byte chunks)
      uint8_t* pcol = pt + sb * C::P_BYTES + (kq >> 6) * N * 128 + 2 * (kq & 7);
      const int pu = (kq & 63) >> 3;
#pragma unroll
      for (int n = 0; n < N; ++n)
        *reinterpret_cast<uint16_t*>(pcol + n * 128 + swz(pu, n)) =
            static_cast<uint16_t>((n & 1) ? (pk[n / 2] >> 16) : (pk[n / 2] & 0xFFFFu));
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok && n_stages >= 1) ok = mbar_wait(&pv_done[(n_stages - 1) & 1], ((n_stages - 1) >> 1) & 1);
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
  }
  __syncthreads();  // every role is done; s_bad / s_timeout are final
  if (warp < 4) {
    // ---- epilogue: row sums and corrections over all keys -> output ----
    const int kq = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      float t = l[n], z = zc[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        t += __shfl_xor_sync(0xffffffffu, t, o);
        z += __shfl_xor_sync(0xffffffffu, z, o);
      }
      if (lane == 0) {
        xch[warp * 64 + n] = t;
        xch2[warp * 64 + n] = z;
      }
    }
    bar_sync_n(1, 128);
    const bool poisoned = s_bad != 0 || s_timeout != 0;
    float* linv = alpha_sm;
    float* zrow = m_next;
    if (kq < R) {
      const int n = kq;
      const float lt = (xch[n] + xch[64 + n]) + (xch[128 + n] + xch[192 + n]);
      zrow[n] = (xch2[n] + xch2[64 + n]) + (xch2[128 + n] + xch2[192 + n]);
      const long long row = static_cast<long long>(si.t0 + n / a.G) * a.Hq + g * a.G + n % a.G;
      if (si.nparts == 1) {
        rowoff[n] = row * D;
        linv[n] = (poisoned || !(lt > 0.f)) ? 0.f : 1.f / lt;
      } else {
        rowoff[n] = (prow(row, si, a.Hq) * a.num_parts + p) * D;
        a.pm[prow(row, si, a.Hq) * a.num_parts + p] = m_sm[n];
        a.pl[prow(row, si, a.Hq) * a.num_parts + p] = poisoned ? -1.f : lt;
      }
    }
    bar_sync_n(1, 128);
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
      float o[16];
      tmem_ld16(tm_o + 16 * c + lane_off, o);
      if (si.nparts > 1) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (16 * c + e < R) a.po[rowoff[16 * c + e] + kq] = o[e] - zrow[16 * c + e];
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (16 * c + e < R)
            store_out(a.out, a.out_dtype, rowoff[16 * c + e] + kq, (o[e] - zrow[16 * c + e]) * linv[16 * c + e]);
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
