// pa_partition_tc.cuh — split-KV partition kernel on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), for 16-bit KV caches and
// up to 64 query rows per KV head (T_b x G, e.g. 8 verify tokens x 8 GQA
// heads), where the QK^T / PV contractions outgrow warp-level mma.
//
// Same contract as pa_partition_mma: one CTA per (partition, KV head,
// sequence); every page of the partition is read once for all rows; per-token
// partials (or the final output when one partition covers the sequence).
//
// Warp roles (128 threads):
//   warps 0, 1  softmax: thread r owns query row r (TMEM lane r)
//   warp 2      MMA issuer (one thread)
//   warp 3      TMA producer (block-table lookup + tile loads, as in the mma path)
// Per 64-key stage s:
//   S(s)  = Q . K_s^T          tcgen05.mma M=128 (rows 0..63 real), N=64, K=D,
//                              A = Q from TMEM, K as K-major B from smem        -> TMEM
//   P(s)  = 2^(S*scale*log2e - m)  (softmax warps, bf16/f16, written to TMEM)
//   O    += P(s) . V_s          tcgen05.mma M=128, N=D, K=64, A = P from TMEM,
//                              V as MN-major B from shared memory             -> TMEM
// Q and P live in tensor memory so shared memory holds only the KV ring (six
// 32 KB stages): a stage is held from its TMA landing until its PV
// completes, and the ring depth beyond that is what keeps HBM busy.
// S(s+1) is issued before PV(s) so the tensor cores work while the softmax
// runs.  The running max is kept lazily: O is rescaled (TMEM load/store) only
// when a row's max grows by more than 2^8, otherwise weights are taken
// relative to the stale max (they stay <= 256, exact enough in 16 bits).
#pragma once

#include "pa_tcgen05.cuh"

namespace pa {

template <int D, int KV>
struct TcCfg {
  static_assert(KV == KV_BF16 || KV == KV_F16, "tensor-memory path takes 16-bit caches");
  static_assert(D == 64 || D == 128, "tensor-memory path: head_dim 64 or 128");
  static constexpr bool kBf16 = (KV == KV_BF16);
  static constexpr int ROWS = 64;                 // real query rows (TMEM lanes 0..63)
  static constexpr int M = 128;                   // MMA rows (64..127 are zero padding)
  static constexpr int SK = 64;                   // keys per stage (= N of the score MMA)
  static constexpr int CH = D / 64;               // 128-byte chunks per key row
  static constexpr int TILE = SK * D * 2;         // one K (or V) stage tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int FIXED = 4 * kMaxPagesPerCta + 512 + 1024;
  static constexpr int NS_FIT = (226 * 1024 - FIXED) / STAGE;
  static constexpr int NS = NS_FIT > 16 ? 16 : NS_FIT;
  static constexpr int BLK_OFF = NS * STAGE;
  static constexpr int BAR_OFF = BLK_OFF + 4 * kMaxPagesPerCta;
  static constexpr int BYTES = BAR_OFF + 512 + 1024;
  // TMEM columns: O [0, D), S buffers [D, D + 2 SK), P buffers (16-bit
  // pairs) [D + 2 SK, D + 3 SK), Q (16-bit pairs) [D + 3 SK, D + 3 SK + D/2)
  static constexpr int S_COL = D;
  static constexpr int P_COL = D + 2 * SK;
  static constexpr int Q_COL = D + 3 * SK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = tc_idesc(M, SK, kBf16, false);
  static constexpr uint32_t IDESC_PV = tc_idesc(M, D, kBf16, true);
  static_assert(NS >= 4, "pipeline needs a few stages");
  static_assert(Q_COL + D / 2 <= TMEM_COLS, "tensor-memory budget");
};

// GATHER (pages of 1, 2 or 4 tokens): four more warps (4..7, one per SM
// sub-partition) fetch key rows with 16-byte cp.async copies instead of TMA
// boxes, block ids looked up per key; warp 3 has no role.  Everything
// downstream of the stage ring is the same kernel.
template <int D, int KV, bool TREE = false, bool GATHER = false>
__global__ void __launch_bounds__(GATHER ? 128 + 32 * kGatherWarps : 128, 1)
    pa_partition_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const PartArgs a) {
  using C = TcCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* blk = reinterpret_cast<int32_t*>(smem + C::BLK_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;                 // [NS] TMA landed
  uint64_t* empty = full + C::NS;        // [NS] stage consumed (MMA commit after PV)
  uint64_t* s_full = empty + C::NS;      // [2] S buffer written (MMA commit)
  uint64_t* s_free = s_full + 2;         // [2] S buffer read (2 softmax warps)
  uint64_t* p_full = s_free + 2;         // [2] P buffer written (2 softmax warps)
  uint64_t* pv_done = p_full + 2;        // [2] PV of the stage using that P buffer done (MMA commit)
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // While the previous kernel may still be running (programmatic dependent
  // launch), warm L2 with the sequence metadata and this partition's
  // block-table slice (prefetches only: every value the kernel uses is
  // loaded after griddepcontrol.wait).
  if (!GATHER && warp == 3 && a.window == 0) {
    if (lane == 0) {
      prefetch_l2(a.begins + b);
      prefetch_l2(a.past_lens + b);
    }
    const long long lpg = (static_cast<long long>(p) * a.part_tokens) >> a.ps_log2;
    const int n = static_cast<int>(min(static_cast<long long>(a.part_tokens >> a.ps_log2),
                                       max(0LL, static_cast<long long>(a.max_blocks) - lpg)));
    for (int j = 32 * lane; j < n; j += 32 * 32) prefetch_l2(a.block_tables + static_cast<size_t>(b) * a.max_blocks + lpg + j);
  }
  // Set-up that reads no input -- barriers, tensor memory, the tensor maps'
  // descriptors -- also runs before the wait.
  if (threadIdx.x == 96) {
    s_bad = 0;
    s_timeout = 0;
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], GATHER ? kGatherWarps : 1);
      mbar_init(&empty[s], 1);
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
  if (!GATHER && warp == 3 && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  tc_fence_before();
  __syncthreads();  // barriers and the TMEM address published
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  // Without a window a partition's first page is p * part_tokens / page_size
  // whatever the sequence's length, so the producer starts fetching its
  // block-table slice before the sequence's bounds are known.
  const bool prefetch = (!GATHER && warp == 3 && a.window == 0);
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
  }
  if (si.err || si.T <= 0 || p >= si.nparts) {
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);  // nothing has used it
    return;
  }

  const int kstart = si.kbase + p * a.part_tokens;
  const int kend = min(kstart + a.part_tokens, si.khi + 1);
  const int lp0 = kstart >> a.ps_log2;
  const int npages = ((kend - 1) >> a.ps_log2) - lp0 + 1;
  const int n_stages = (kend - kstart + C::SK - 1) / C::SK;
  const int R = si.T * a.G;

  // ---- the producer starts while warps 0-1 stage Q ----
  if (warp < 3) {
    if (warp < 2) {
      // Q rows into TMEM (lane = query row r = token r/G, head g*G + r%G; two
      // 16-bit elements per column), lanes R..63 zero.  Lanes 64..127 are
      // left as they are: they only feed S, P and O rows nobody reads.
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
    bar_sync_n(2, 96);  // Q is in place for the MMA warp
    tc_fence_after();
  }
  const uint32_t tm_o = tmem;                      // O
  const uint32_t tm_s0 = tmem + C::S_COL;          // S buffers
  const uint32_t tm_p0 = tmem + C::P_COL;          // P buffers (16-bit pairs)
  const uint32_t tm_q = tmem + C::Q_COL;           // Q (16-bit pairs)

  if (GATHER && warp >= 4) {
    // ======================= cp.async gather producers ======================
    // Warp 4 + pw copies key rows [16 pw, 16 pw + 16) of every stage.  Lane
    // (h, u): 16-byte unit u of key row h of each group of KPI rows, so one
    // warp instruction copies KPI whole rows (256 or 128 contiguous bytes
    // each).  A warp's copies of one stage form one group; the warp arrives
    // on the stage's barrier once that group has landed, DEPTH groups behind
    // its newest, so DEPTH + 1 stages are in flight and the ring keeps two
    // more for the consumers (the stage whose PV is pending and the next
    // one's scores).  Block ids are loaded two stages ahead and checked only
    // when used, so no load latency sits between two stages' copies.
    constexpr int UPK = D * 2 / 16;  // 16-byte units per key row
    constexpr int KPI = 32 / UPK;    // key rows per warp instruction
    constexpr int ROWS_W = C::SK / kGatherWarps;
    constexpr int DEPTH = (C::NS - 3) < 5 ? (C::NS - 3) : 5;
    static_assert(DEPTH >= 2, "the ring must hold the stages in flight plus two being consumed");
    static_assert(ROWS_W <= 32 && ROWS_W % KPI == 0, "one id per lane covers a warp's rows");
    const int pw = warp - 4;
    const int u = lane % UPK, h = lane / UPK;
    const int c = u >> 3, w = u & 7;
    const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
    const uint64_t blk_bytes = static_cast<uint64_t>(a.Hkv) * a.ps * D * 2;
    const uint8_t* kb = a.k_bytes + static_cast<size_t>(g) * a.ps * D * 2 + 16 * u;
    const uint8_t* vb = a.v_bytes + static_cast<size_t>(g) * a.ps * D * 2 + 16 * u;
    int bad = 0;
    // raw id of key row `lane` of this warp's slice (0 past the partition)
    auto load_id = [&](int s) -> int {
      const int k = kstart + s * C::SK + pw * ROWS_W + lane;
      return (lane < ROWS_W && k < kend) ? __ldg(bt + (k >> a.ps_log2)) : 0;
    };
    int na = load_id(0), nb = load_id(1);  // ids of the next stage and of the one after
    int issued = 0;
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % C::NS;
      if (s >= C::NS && !mbar_wait(&empty[slot], ((s / C::NS) - 1) & 1)) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        break;
      }
      int idl = na;
      na = nb;
      if (s + 2 < n_stages) nb = load_id(s + 2);
      if (static_cast<unsigned>(idl) >= static_cast<unsigned>(a.num_blocks)) {
        bad = 1;
        idl = 0;
      }
      const int key0 = kstart + s * C::SK;
      uint8_t* st = smem + slot * C::STAGE;
#pragma unroll
      for (int i = 0; i < ROWS_W / KPI; ++i) {
        const int r = i * KPI + h;        // row within this warp's slice
        const int kl = pw * ROWS_W + r;   // key row within the stage
        const int id = __shfl_sync(0xffffffffu, idl, r);
        const int key = key0 + kl;
        const uint64_t src = static_cast<uint64_t>(id) * blk_bytes + static_cast<uint32_t>(key & (a.ps - 1)) * (D * 2);
        // tile layout [chunk][key][128 B], 16-byte units swizzled by key & 7
        const uint32_t dst = static_cast<uint32_t>((c * C::SK + kl) * 128 + ((w ^ (kl & 7)) << 4));
        const uint32_t n = key < kend ? 16u : 0u;  // past the partition: zeros
        cp_async16(st + dst, kb + src, n);
        cp_async16(st + C::TILE + dst, vb + src, n);
        if (a.trace != nullptr && u == 0 && key < kend && (key & (a.ps - 1)) == 0)
          atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + (key >> a.ps_log2), id + 1);
      }
      cp_async_commit();
      issued = s + 1;
      if (s >= DEPTH) {
        cp_async_wait_group<DEPTH>();
        fence_proxy_async();  // the copies, seen by the tensor cores' proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[(s - DEPTH) % C::NS]);
      }
    }
    cp_async_wait_all();
    fence_proxy_async();
    // the flag is set before the last stages are published, so the softmax
    // warps see it once their last PV has completed
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      s_bad = 1;
      atomicOr(a.status, PA_STATUS_BLOCK_ID);
    }
    __syncwarp();
    if (lane == 0)
      for (int q = max(0, issued - DEPTH); q < issued; ++q) mbar_arrive(&full[q % C::NS]);
  } else if (GATHER && warp == 3) {
    // no role in the gather variant
  } else if (warp == 3) {
    // =========================== TMA producer ===============================
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
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % C::NS;
      if (s >= C::NS && !mbar_wait(&empty[slot], ((s / C::NS) - 1) & 1)) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        break;
      }
      const int key0 = kstart + s * C::SK;
      const int nk = min(C::SK, kend - key0);
      const int nseg = (nk + br - 1) >> br_log2;
      uint8_t* st = smem + slot * C::STAGE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nseg * br * D * 2 * 2));
      __syncwarp();
      for (int j = lane; j < nseg * C::CH; j += 32) {
        const int seg = j / C::CH, c = j % C::CH;
        const int key = key0 + (seg << br_log2);
        const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
        const int id = blk[lp - lp0];
        // tile layout [chunk][key][128 B]: rows of one chunk are contiguous
        const uint32_t off = static_cast<uint32_t>((c * C::SK + (seg << br_log2)) * 128);
        tma_load_4d(st + off, &tmK, c * 64, slot0, g, id, &full[slot]);
        tma_load_4d(st + C::TILE + off, &tmV, c * 64, slot0, g, id, &full[slot]);
        if (a.trace != nullptr && c == 0 && slot0 == 0)
          atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
      }
    }
  } else if (warp == 2) {
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
    const int r = warp * 32 + lane;                          // TMEM lane / query row
    const int rc = min(r, R - 1);                            // padding rows mask like the last row
    // with a tree mask the row sees the new tokens its mask names (hi covers
    // them all); without one, the causal chain up to its own position
    // (TREE: the launcher picks this instantiation when a mask is given)
    const int hi = TREE ? si.L + si.T - 1 : si.L + rc / a.G;
    const int clean_hi = TREE ? si.L - 1 : hi;
    const uint32_t tmask = TREE ? row_new_token_mask(a.tree_mask, si.t0 + rc / a.G, rc / a.G) : 0u;
    const int lo = a.window > 0 ? si.L + rc / a.G - a.window + 1 : INT_MIN;
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
      float x[C::SK];  // raw scores q.k (the scale is applied inside the exponent)
      tmem_ld64(tm_s0 + sb * C::SK + lane_off, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);

      const int key0 = kstart + s * C::SK;
      const bool clean = key0 >= lo && key0 + C::SK - 1 <= clean_hi;
      // The stage's 64 keys as one validity mask per row (inside [lo, hi],
      // and with a tree mask a past key or a new token the mask names), so
      // the unrolled loop below tests one constant bit per key.
      uint64_t vmask = ~0ull;
      if (!clean) {
        const long long a0 = max(0LL, static_cast<long long>(lo) - key0);
        const long long b0 = min(63LL, static_cast<long long>(hi) - key0);
        vmask = (a0 > b0) ? 0ull : ((b0 - a0 == 63) ? ~0ull : (((1ull << (b0 - a0 + 1)) - 1ull) << a0));
        if constexpr (TREE) {
          const long long sh = static_cast<long long>(si.L) - key0;  // bit of new token 0
          const uint64_t past = sh <= 0 ? 0ull : (sh >= 64 ? ~0ull : ((1ull << sh) - 1ull));
          const uint64_t named = (sh >= 64 || sh <= -64) ? 0ull
                                 : (sh >= 0 ? (static_cast<uint64_t>(tmask) << sh)
                                            : (static_cast<uint64_t>(tmask) >> -sh));
          vmask &= past | named;
        }
#pragma unroll
        for (int j = 0; j < C::SK; ++j) x[j] = ((vmask >> j) & 1ull) ? x[j] : -INFINITY;
      }
      // row max in four independent chains; scaling by sl2 > 0 commutes
      // with the max (-inf stays -inf)
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < C::SK; ++j) m4[j & 3] = fmaxf(m4[j & 3], x[j]);
      const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
      // lazy running max: move the reference only when the row max grows by
      // more than 2^8 (or on the first finite score)
      const bool need = (mt > m_ref + 8.f) || (m_ref == -INFINITY && mt != -INFINITY);
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? ex2(m_ref - m_new) : 1.f;  // 0 when m_ref was -inf
      if (__any_sync(0xffffffffu, need) && s >= 1) {
        // rescale this warp's O rows once the previous PV has landed
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
      m_ref = m_new;
      const float nmu = (m_ref == -INFINITY) ? 0.f : -m_ref;
      uint32_t pk[C::SK / 2];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < C::SK; j += 2) {
        const float p0 = ex2_free(fmaf(x[j], sl2, nmu)), p1 = ex2_free(fmaf(x[j + 1], sl2, nmu));
        l4[(j >> 1) & 3] += p0 + p1;
        pk[j / 2] = pack2<C::kBf16>(p0, p1);
      }
      l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
      // the P buffer is free once the PV two stages back has finished
      if (s >= 2 && !mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1)) {
        ok = false;
        break;
      }
      tmem_st32(tm_p0 + sb * (C::SK / 2) + lane_off, reinterpret_cast<const float*>(pk));
      // V rows of keys outside every row's range may hold garbage (even NaN);
      // their weights are 0 but 0 * NaN is not: clear those rows.
      // Thread k clears key row k (the 64 softmax threads cover the stage),
      // its 16-byte units in an order rotated by k so that the eight threads
      // of a store phase hit eight different bank groups.
      static_assert(C::SK == 64, "one softmax thread per key row of the stage");
      if (key0 < si.klo || key0 + C::SK - 1 > si.khi) {
        const int k = threadIdx.x;
        const int key = key0 + k;
        if (key < si.klo || key > si.khi) {
          uint8_t* vrow = smem + (s % C::NS) * C::STAGE + C::TILE + k * 128;
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(vrow + c * C::SK * 128 + 16 * ((u + k) & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    // ---- epilogue: O row from TMEM -> partial or output ----
    if (ok && n_stages >= 1 && !mbar_wait(&pv_done[(n_stages - 1) & 1], ((n_stages - 1) >> 1) & 1)) ok = false;
    if (!ok) {
      if (lane == 0) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    tc_fence_after();
    const bool poisoned = s_bad != 0 || s_timeout != 0 || !ok;
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
          for (int e = 0; e < 32; ++e) store_out(a.out, a.out_dtype, row * D + 32 * c + e, poisoned ? 0.f : o[e] * inv);
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
