// pa_partition_tk.cuh — split-KV partition kernel on the 5th-generation tensor
// cores with the keys of a stage on the MMA's M dimension ("transposed"
// scores), for 16-bit KV caches, head_dim 64 / 128, up to 64 query rows per KV
// head (T_b x G).
//
// Same contract as the other partition kernels (OpenVINO issue 38153, the
// verify step of speculative decoding over a paged cache: one CTA per
// (partition, KV head, sequence); every page of the partition is read once for
// all rows; per-token partials, or the final output when one partition covers
// the sequence).
//
// Per 128-key stage s (query rows n < N, N = 16 / 32 / 64 >= T_b x G):
//   S^T(s) = K_s . Q^T           M = 128 keys, N rows, K = D.  A = K tile
//                                (K-major, smem), B = Q tile (K-major, smem)   -> TMEM
//   P^T(s) = 2^(S^T scale log2e - m_n)   softmax warps: thread = key = TMEM lane
//   O^T   += V_s^T . P^T(s)      M = 128 (head dim), N rows, K = 128 keys.  A =
//                                V tile read MN-major, B = P^T (MN-major, smem) -> TMEM
// A softmax thread owns one key and the N rows of it, so a stage costs a
// thread N exponentials: the work follows the real row count instead of a
// fixed 128-row tile, and no per-row reduction is needed on the common path.
// The running max is kept lazily per row (weights are taken relative to a
// stale max until some score exceeds it by 2^8); the four softmax warps agree
// on "does any row need a new max" with one barrier-reduction per stage, and
// only then exchange row maxima through shared memory and rescale O^T.
//
// Warp roles (192 threads):
//   warps 0..3  softmax: warp w owns TMEM lanes 32w..32w+31 (keys of S^T, head
//               dims of O^T); also stage Q and write the epilogue
//   warp 4      MMA issuer (one thread)
//   warp 5      TMA producer: block-table lookup, K and V tiles
// Shared-memory ring: K and V tiles of consecutive stages (K_0 V_0 K_1 V_1 ...);
// a K tile is released when its S^T MMAs complete, a V tile when its PV does.
#pragma once

#include "pa_partition_tc.cuh"

namespace pa {

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// N consecutive 32-bit columns of this thread's TMEM lane (N = 16 / 32 / 64).
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float* v) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32(taddr + 32 * c, v + 32 * c);
  }
}

// Instruction descriptor, kind::f16, f32 accumulation, optional MN-major A / B.
__host__ __device__ constexpr uint32_t tk_idesc(int M, int N, bool bf16, bool a_mn_major, bool b_mn_major) {
  return tc_idesc(M, N, bf16, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// Tensor-memory columns (a power of two >= 32) for O^T and two S^T buffers.
__host__ __device__ constexpr int tk_tmem_cols(int n) { return 3 * n <= 32 ? 32 : (3 * n <= 64 ? 64 : (3 * n <= 128 ? 128 : 256)); }

template <int D, int KV, int N>
struct TkCfg {
  static_assert(KV == KV_BF16 || KV == KV_F16, "16-bit caches");
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(N == 16 || N == 32 || N == 64, "row tile 16 / 32 / 64");
  static constexpr bool kBf16 = (KV == KV_BF16);
  static constexpr int SK = 128;                      // keys per stage (= M of the score MMA)
  static constexpr int CH = D / 64;                   // 128-byte chunks of a key row
  static constexpr int TILE = SK * D * 2;             // one K or V tile, [chunk][key][128 B]
  static constexpr int Q_BYTES = N * D * 2;           // Q tile, [chunk][row][128 B]
  static constexpr int P_BYTES = SK * 128;            // P^T tile, [key][64 row slots x 2 B]
  static constexpr int MISC = 3072;                   // barriers, row maxima, exchange
  static constexpr int FIXED = Q_BYTES + 2 * P_BYTES + 4 * kMaxPagesPerCta + MISC + 1024;
  static constexpr int NS_FIT = (226 * 1024 - FIXED) / TILE;
  static constexpr int NS = NS_FIT > 16 ? 16 : NS_FIT;  // K / V tiles in the ring
  static constexpr int Q_OFF = NS * TILE;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int BLK_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int MISC_OFF = BLK_OFF + 4 * kMaxPagesPerCta;
  static constexpr int BYTES = MISC_OFF + MISC + 1024;
  static constexpr int TMEM_COLS = tk_tmem_cols(N);   // O^T [0, N), S^T buffers [N, 3N)
  static constexpr uint32_t IDESC_S = tk_idesc(128, N, kBf16, false, false);
  static constexpr uint32_t IDESC_PV = tk_idesc(128, N, kBf16, true, true);
  static_assert(NS >= 4, "ring needs a few tiles");
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0, "swizzled tiles are 1024-aligned");
};

template <int D, int KV, int N>
__global__ void __launch_bounds__(192, 1)
    pa_partition_tk(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const PartArgs a) {
  using C = TkCfg<D, KV, N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qt = smem + C::Q_OFF;
  uint8_t* pt = smem + C::P_OFF;
  int32_t* blk = reinterpret_cast<int32_t*>(smem + C::BLK_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::MISC_OFF);
  uint64_t* full = bars;                 // [NS] tile landed (TMA)
  uint64_t* empty = full + C::NS;        // [NS] tile consumed (MMA commit)
  uint64_t* s_full = empty + C::NS;      // [2] S^T buffer written (MMA commit)
  uint64_t* s_free = s_full + 2;         // [2] S^T buffer read (4 softmax warps)
  uint64_t* p_full = s_free + 2;         // [2] P^T buffer written (4 softmax warps)
  uint64_t* pv_done = p_full + 2;        // [2] PV that read that P^T buffer done (MMA commit)
  float* m_sm = reinterpret_cast<float*>(smem + C::MISC_OFF + 512);   // [64] row reference maxima
  float* xch = m_sm + 64;                                             // [4][64] per-warp row values
  float* m_next = xch + 256;                                          // [64] new reference maxima
  float* alpha_sm = m_next + 64;                                      // [64] their rescale factors
  long long* rowoff = reinterpret_cast<long long*>(alpha_sm + 64);    // [64] epilogue: output offsets
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  // Without a window a partition's first page is p * part_tokens / page_size
  // whatever the sequence's length, so the producer starts fetching its
  // block-table slice before the sequence's bounds are known.
  const bool prefetch = (warp == 5 && a.window == 0);
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
    if (prefetch) cp_async_wait_all();  // no copy into shared memory outlives the CTA
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

  // ---- set-up: barriers; then the producer starts while the others
  // allocate tensor memory and stage Q ----
  if (threadIdx.x == 160) {
    s_bad = 0;
    s_timeout = 0;
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
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
    // Q rows -> K-major swizzled tile (row n = token n/G, head g*G + n%G);
    // rows R..N-1 are zero.
    for (int idx = threadIdx.x; idx < N * (D / 8); idx += 128) {
      const int n = idx / (D / 8), u16 = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < R) {
        const size_t row = static_cast<size_t>(si.t0 + n / a.G) * a.Hq + g * a.G + n % a.G;
        v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + row * D) + u16);
      }
      *reinterpret_cast<uint4*>(qt + ((u16 >> 3) * N + n) * 128 + swz(u16 & 7, n)) = v;
    }
    if (threadIdx.x < 64) m_sm[threadIdx.x] = -INFINITY;
    fence_proxy_async();  // the Q tile is read by the tensor cores
  }
  if (warp < 5) {
    // TMEM address and Q tile published to the softmax and MMA warps
    tc_fence_before();
    bar_sync_n(2, 160);
    tc_fence_after();
    tmem = s_tmem;
  }
  const uint32_t tm_o = tmem;            // O^T: lane = head dim, column = row
  const uint32_t tm_s0 = tmem + N;       // S^T buffers: lane = key, column = row

  if (warp == 5) {
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
    const int items = 2 * n_stages;
    int issued = 0;
    for (int i = 0; i < items; ++i, ++issued) {
      const int slot = i % C::NS, s = i >> 1;
      const bool is_v = (i & 1) != 0;
      if (i >= C::NS && !mbar_wait(&empty[slot], ((i / C::NS) - 1) & 1)) {
        ok = false;
        break;
      }
      const int key0 = kstart + s * C::SK;
      const int nk = min(C::SK, kend - key0);
      const int nseg = (nk + br - 1) >> br_log2;
      uint8_t* tile = smem + slot * C::TILE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nseg * br * D * 2));
      __syncwarp();
      for (int j = lane; j < nseg * C::CH; j += 32) {
        const int seg = j / C::CH, c = j % C::CH;
        const int key = key0 + (seg << br_log2);
        const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
        const int id = blk[lp - lp0];
        const uint32_t off = static_cast<uint32_t>((c * C::SK + (seg << br_log2)) * 128);
        tma_load_4d(tile + off, is_v ? &tmV : &tmK, c * 64, slot0, g, id, &full[slot]);
        if (!is_v && a.trace != nullptr && c == 0 && slot0 == 0)
          atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
      }
    }
    // leave no copy in flight: the last tiles issued have landed
    if (lane == 0) {
      for (int i = max(0, issued - C::NS); i < issued; ++i)
        if (!mbar_wait(&full[i % C::NS], (i / C::NS) & 1)) ok = false;
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else if (warp == 4) {
    // =========================== MMA issuer =================================
    if (lane == 0) {
      const uint32_t q_base = smem_u32(qt);
      auto issue_pv = [&](int s) -> bool {
        const int vi = 2 * s + 1, vslot = vi % C::NS, pb = s & 1;
        if (!mbar_wait(&full[vslot], (vi / C::NS) & 1)) return false;
        if (!mbar_wait(&p_full[pb], (s >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(smem + vslot * C::TILE);
        const uint32_t p_base = smem_u32(pt + pb * C::P_BYTES);
#pragma unroll
        for (int j = 0; j < C::SK / 16; ++j) {
          const uint64_t ad = sw128_desc(v_base + j * 16 * 128, D == 128 ? C::SK * 128 : 0, 1024);
          const uint64_t bd = sw128_desc(p_base + j * 16 * 128, 0, 1024);
          tc_mma(tm_o, ad, bd, C::IDESC_PV, (s > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[pb]);
        tc_commit(&empty[vslot]);
        return true;
      };
      for (int s = 0; s < n_stages && ok; ++s) {
        const int ki = 2 * s, kslot = ki % C::NS, sb = s & 1;
        if (!mbar_wait(&full[kslot], (ki / C::NS) & 1) ||
            (s >= 2 && !mbar_wait(&s_free[sb], ((s >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(smem + kslot * C::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk >> 2, w = kk & 3;
          const uint64_t ad = sw128_desc(k_base + c * C::SK * 128 + 32 * w, 16, 1024);
          const uint64_t bd = sw128_desc(q_base + c * N * 128 + 32 * w, 16, 1024);
          tc_mma(tm_s0 + sb * N, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        tc_commit(&empty[kslot]);
        if (s >= 1) ok = issue_pv(s - 1);
      }
      if (ok && n_stages >= 1) ok = issue_pv(n_stages - 1);
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  }

  // =========================== softmax warps (keys) ==========================
  // Thread kq owns key kq of every stage (TMEM lane kq of S^T) and head dim
  // kq of O^T.  Each loop iteration runs the same barriers on all four warps,
  // also after a wait has timed out, so the named barriers always complete.
  float l[N];
  if (warp < 4) {
    const int kq = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale_log2;
#pragma unroll
    for (int n = 0; n < N; ++n) l[n] = 0.f;
    for (int s = 0; s < n_stages; ++s) {
      const int sb = s & 1;
      if (ok) ok = mbar_wait(&s_full[sb], (s >> 1) & 1);
      tc_fence_after();
      float v[N];
      tmem_ld_n<N>(tm_s0 + sb * N + lane_off, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);

      // rows n for which this key is in range: n in [nlo, nhi)
      const int key0 = kstart + s * C::SK, key = key0 + kq;
      const int dk = key - si.L;
      const int nlo = dk > 0 ? dk * a.G : 0;
      int nhi = R;
      if (a.window > 0) nhi = min(R, max(0, (dk + a.window) * a.G));
      const bool clean = (nlo == 0 && nhi >= R);
      bool need = false;
#pragma unroll
      for (int n4 = 0; n4 < N; n4 += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_sm + n4);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = n4 + e;
          float x = v[n] * sl2;
          if (!clean) x = (n >= nlo && n < nhi) ? x : -INFINITY;
          v[n] = x;
          need |= x > mm[e] + 8.f;
        }
      }
      if (bar_any(1, 128, need)) {
        // ---- a row's max grew by more than 2^8 (or first scores): new references ----
#pragma unroll
        for (int n = 0; n < N; ++n) {
          float t = v[n];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
          if (lane == 0) xch[warp * 64 + n] = t;
        }
        bar_sync_n(1, 128);
        // references move only for rows whose max grew by more than 2^8
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const float rm = fmaxf(fmaxf(xch[n], xch[64 + n]), fmaxf(xch[128 + n], xch[192 + n]));
          const float mo = m_sm[n];
          const float mn = rm > mo + 8.f ? rm : mo;
          const float al = (mn == mo) ? 1.f : ex2(mo - mn);
          l[n] *= al;
          if (n == threadIdx.x) {
            m_next[n] = mn;
            alpha_sm[n] = al;
          }
        }
        bar_sync_n(1, 128);  // every thread has read m_sm / xch; m_next / alpha_sm are written
        if (threadIdx.x < N) m_sm[threadIdx.x] = m_next[threadIdx.x];
        if (s >= 1) {
          // rescale O^T once the previous PV has landed
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
        bar_sync_n(1, 128);  // m_sm published
      }
      // weights, packed two rows per 32-bit word
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
          pk[(n4 + e) / 2] = pack2<C::kBf16>(p0, p1);
        }
      }
      // the P^T buffer is free once the PV two stages back has finished
      if (s >= 2 && ok) ok = mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1);
      uint8_t* prow = pt + sb * C::P_BYTES + kq * 128;
#pragma unroll
      for (int u = 0; u < N / 8; ++u)
        *reinterpret_cast<uint4*>(prow + swz(u, kq)) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      // V rows of keys outside every row's range may hold garbage (even NaN):
      // their weights are 0, but 0 * NaN is not, so clear them once landed.
      if (key0 < si.klo || key0 + C::SK - 1 > si.khi) {
        const int vi = 2 * s + 1;
        if (ok) ok = mbar_wait(&full[vi % C::NS], (vi / C::NS) & 1);
        if (key < si.klo || key > si.khi) {
          uint8_t* vt = smem + (vi % C::NS) * C::TILE;
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(vt + (c * C::SK + kq) * 128 + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
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
    // ---- epilogue: row sums over all keys, O^T lane (head dim kq) -> output ----
    const int kq = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      float t = l[n];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (lane == 0) xch[warp * 64 + n] = t;
    }
    bar_sync_n(1, 128);
    const bool poisoned = s_bad != 0 || s_timeout != 0;
    // one thread per row: where the row goes, and its normaliser
    float* linv = alpha_sm;
    if (kq < R) {
      const int n = kq;
      const float lt = (xch[n] + xch[64 + n]) + (xch[128 + n] + xch[192 + n]);
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
      if (kq < D) {
        if (si.nparts > 1) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (16 * c + e < R) a.po[rowoff[16 * c + e] + kq] = o[e];
        } else if (a.out_dtype == PA_BF16) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (16 * c + e < R)
              reinterpret_cast<__nv_bfloat16*>(a.out)[rowoff[16 * c + e] + kq] = __float2bfloat16_rn(o[e] * linv[16 * c + e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (16 * c + e < R) store_out(a.out, a.out_dtype, rowoff[16 * c + e] + kq, o[e] * linv[16 * c + e]);
        }
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
