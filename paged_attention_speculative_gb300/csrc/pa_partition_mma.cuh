// pa_partition_mma.cuh — split-KV partition kernel, tensor-core path
// (16-bit KV caches, and u8 caches dequantised on the fly).
//
// One CTA owns one (KV partition p, KV head g, sequence b).  It streams the
// partition's pages once — for ALL T_b x G query rows of the GQA group (the
// "GQA read-once, 256-token partitions" single-token stage of OpenVINO issue
// 38153, "Cause", kept for T > 1) — and writes per-query-token partials
// (max, denominator, unnormalised output) indexed [token, head, partition]
// (the per-token segment buffer the dual-radeon-vllm article, use_3d section,
// shows must replace a per-sequence one).
//
// Warp roles: warp 4 is the producer — it looks each page up in the block
// table and issues 128-byte-swizzled TMA tile loads of the page's K and V
// rows (plus 1-D bulk copies of u8 scales / zero-points) into a ring of
// NS shared-memory stages guarded by full / empty mbarriers.  Warps 0..3 are
// consumers: each owns a set of query rows (8 or 16) and a share of every
// stage's 16-key chunks, and keeps its own online-softmax state, so no warp
// waits on another inside the loop.  Scores are computed transposed,
// S^T[key, row] = K . Q^T with mma.sync m16n8k16 (keys on M, query rows on N,
// so 1..8 rows waste nothing), P is transposed in registers with movmatrix,
// and O^T[d, row] += V^T . P^T.  The warps' states merge through shared
// memory at the end.
//
// Pages of 1, 2 or 4 tokens (16-bit caches, head_dim 256): no TMA box fits a
// swizzle atom, so two producer warps gather whole rows into rows padded by
// 16 bytes instead of swizzled (the pad spreads the eight rows an ldmatrix
// phase reads over all 32 banks): warp 4 copies each key's K row with a 1-D
// bulk copy of its own (one key per lane, the block id looked up a stage
// ahead), warp 5 its V row with 16-byte cp.async (the warp's 32 lanes on one
// row).  The magik.net article ("The
// Hypothesis: page_size=1 Scatter-Gather") describes this layout: every key
// is its own block-table lookup, and each lookup still feeds whole-row copies.
//
// u8 caches: codes are exact in f16 (code = f16(0x6400 | code) - 1024), so
// q.K = scale_j (q.code_j - zp_j sum(q)) and the value sum is
// sum_j p_j scale_j code_j - sum_j p_j scale_j zp_j — the dequantisation costs
// one FMA per key, not per element.  u8 V pages hold their codes dim-major, so
// a stage segment of V arrives as a [head dim][key] tile (one TMA box) whose
// rows are the A operand of O^T = V^T . P^T as they are; u8 keys are taken in
// their natural order within a 16-key chunk.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D, int KV, bool GATHER = false>
struct MmaCfg {
  static constexpr bool kU8 = (KV == KV_U8);
  static constexpr bool kBf16 = (KV == KV_BF16);       // u8 math runs in f16
  static constexpr int EB = kU8 ? 1 : 2;               // bytes per cache element
  static constexpr int ROW_BYTES = D * EB;             // one key's row
  static constexpr int CHUNKS = ROW_BYTES / 128;       // 128-byte swizzle rows per key
  static constexpr int ELEMS_128 = 128 / EB;           // elements per 128-byte row
  static constexpr int SK = (ROW_BYTES >= 512) ? 32 : 64;  // keys per pipeline stage
  static constexpr int PITCH = GATHER ? ROW_BYTES + 16 : ROW_BYTES;  // bytes between keys' rows
  static constexpr int TILE = SK * PITCH;              // bytes of one K (or V) stage tile
  static constexpr int SZ = kU8 ? SK * 2 : 0;          // one fp16 scale (or zp) array
  // stages start on 1024-byte boundaries: the 128-byte swizzle pattern is a
  // function of the shared-memory address bits 7..9
  static constexpr int STAGE = ((2 * TILE + 4 * SZ) + 1023) / 1024 * 1024;
  static constexpr int NS = (STAGE <= 20 * 1024) ? 5 : 3;  // stages in flight
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;
  static constexpr int CHUNKS_PER_STAGE = SK / 16;
  static_assert(CHUNKS >= 1, "head_dim too small for the swizzled layout");
  static_assert(!(GATHER && kU8), "u8 V pages are dim-major: no per-key gather");
};

template <int D, int KV, int NT, bool GATHER = false>
struct MmaSmem {
  using C = MmaCfg<D, KV, GATHER>;
  static constexpr int RPW = 8 * NT;                   // rows per consumer warp
  static constexpr int CTAS_PER_SM = (NT == 2) ? 1 : 2;  // register budget of the launch bounds
  static constexpr int MERGE_LD = D + 4;
  static constexpr int MERGE_BYTES = kConsumerWarps * RPW * (MERGE_LD + 2) * 4;
  static_assert(MERGE_BYTES <= C::NS * C::STAGE, "merge area must fit in the stage ring");
  static constexpr int BAR_OFF = C::NS * C::STAGE;
  static constexpr int BLK_OFF = BAR_OFF + 2 * C::NS * 8;
  static constexpr int BYTES = BLK_OFF + 4 * kMaxPagesPerCta + 1024;  // + alignment slack
};

// Physical head-dim index of mma row m of m-tile mt in the O^T accumulator.
template <int D, bool kU8>
__device__ __forceinline__ int out_dim(int mt, int m) {
  return 16 * mt + m;
}

template <int D, int KV, int NT, bool TREE = false, bool GATHER = false>
__global__ void __launch_bounds__(GATHER ? kThreads + 32 : kThreads, (NT == 2) ? 1 : 2)
    pa_partition_mma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const PartArgs a) {
  using C = MmaCfg<D, KV, GATHER>;
  using S = MmaSmem<D, KV, NT, GATHER>;
  constexpr bool kBf = C::kBf16;
  constexpr int RPW = S::RPW;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  uint64_t* empty = full + C::NS;
  int32_t* blk = reinterpret_cast<int32_t*>(smem + S::BLK_OFF);
  __shared__ int s_timeout;
  __shared__ int s_bad;

  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Set-up that reads no input -- barriers, the tensor maps' descriptors --
  // runs before the wait, overlapping the previous kernel's tail.
  if (threadIdx.x == 0) {
    s_timeout = 0;
    s_bad = 0;
    for (int s = 0; s < C::NS; ++s) {
      // gather: the producer's lane 0 (K bytes expected) and its 32 lanes'
      // cp.async arrivals (V rows)
      mbar_init(&full[s], GATHER ? 33 : 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  if (!GATHER && warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();  // barriers ready
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  // Without a window a partition's first page is p * part_tokens / page_size
  // whatever the sequence's length, so the producer starts fetching its
  // block-table slice before the sequence's bounds are known.
  const bool prefetch = (!GATHER && warp == kConsumerWarps && a.window == 0);
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
    if (p == 0 && si.rows_ok) {  // leave the sequence's rows of this KV group zero
      const int n = si.T * a.G * D;
      for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        const int t = si.t0 + r / a.G, h = g * a.G + r % a.G;
        store_out(a.out, a.out_dtype, (static_cast<size_t>(t) * a.Hq + h) * D + d, 0.f);
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

  // =========================== producer warp ===============================
  if (warp >= kConsumerWarps) {
    if constexpr (GATHER) {
      const bool vwarp = warp == kConsumerWarps + 1;  // V rows by cp.async; warp kConsumerWarps: K by bulk copy
      // One key per lane: validate its block id (a bad one is reported,
      // clamped to page 0 and the partition's result discarded), then warp 4
      // copies the key's K row whole with a bulk copy and warp 5 the V rows
      // by 16-byte cp.async, all 32 lanes on one row at a time.  Measured at
      // Gemma global T=2, 32k keys, page 1: both rows by bulk copy from one
      // warp 120.0 us (one 512-byte copy per ~36 SM cycles); V by cp.async
      // from the same warp 109.1 us; V from a warp of its own 92.0 us.  The
      // next stage's ids are loaded before this stage waits for its slot.
      static_assert(C::SK == 32 && C::ROW_BYTES == 512, "gather layout: one key per lane, 32 units per row");
      constexpr int KPL = (C::SK + 31) / 32;  // keys per lane and stage
      const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
      int idn[KPL];
#pragma unroll
      for (int u = 0; u < KPL; ++u) {
        const int key = kstart + lane + 32 * u;
        idn[u] = (lane + 32 * u < C::SK && key < kend) ? __ldg(bt + (key >> a.ps_log2)) : 0;
      }
      int issued = 0;
      bool ok = true;
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % C::NS;
        const int key0 = kstart + s * C::SK;
        const int nk = min(C::SK, kend - key0);
        int id[KPL];
        int bad = 0;
#pragma unroll
        for (int u = 0; u < KPL; ++u) {
          id[u] = idn[u];
          if (lane + 32 * u < nk && static_cast<unsigned>(id[u]) >= static_cast<unsigned>(a.num_blocks)) {
            bad = 1;
            id[u] = 0;
          }
          const int nkey = key0 + C::SK + lane + 32 * u;
          idn[u] = (lane + 32 * u < C::SK && nkey < kend) ? __ldg(bt + (nkey >> a.ps_log2)) : 0;
        }
        if (!vwarp && __any_sync(0xffffffffu, bad) && lane == 0) {
          s_bad = 1;  // published to the consumers by this stage's full-barrier arrive
          atomicOr(a.status, PA_STATUS_BLOCK_ID);
        }
        if (s >= C::NS && !mbar_wait(&empty[slot], ((s / C::NS) - 1) & 1)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + slot * C::STAGE;
        const int j = lane;
        const size_t off = ((static_cast<size_t>(id[0]) * a.Hkv + g) * a.ps + ((key0 + j) & (a.ps - 1))) * C::ROW_BYTES;
        if (!vwarp) {
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nk * C::ROW_BYTES));
          __syncwarp();
          if (j < nk) {
            bulk_load(st + j * C::PITCH, a.k_bytes + off, C::ROW_BYTES, &full[slot]);
            if (a.trace != nullptr && ((key0 + j) & (a.ps - 1)) == 0)
              atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + ((key0 + j) >> a.ps_log2),
                        id[0] + 1);
          }
        } else {
          // V: row k's unit `lane`, row offsets passed along the warp
          for (int k = 0; k < nk; ++k) {
            const size_t roff = __shfl_sync(0xffffffffu, off, k);
            cp_async16(st + C::TILE + k * C::PITCH + 16 * lane, a.v_bytes + roff + 16 * lane, 16);
          }
          cp_async_mbar_arrive_noinc(&full[slot]);
        }
        issued = s + 1;
      }
      if (!ok) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        for (int s = max(0, issued - C::NS); s < issued; ++s) mbar_wait(&full[s % C::NS], (s / C::NS) & 1);
      }
      return;
    } else {
      // Stage this partition's block ids in one coalesced pass and validate
      // them.  A bad id is reported, clamped to page 0 (so every copy stays in
      // bounds) and the partition's result is discarded after the loop.
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
        s_bad = 1;  // published to the consumers by the first full-barrier arrive
        atomicOr(a.status, PA_STATUS_BLOCK_ID);
      }
      __syncwarp();
      const int br_log2 = a.box_log2;
      const int br = 1 << br_log2;
      int issued = 0;
      bool ok = true;
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % C::NS;
        if (s >= C::NS && !mbar_wait(&empty[slot], ((s / C::NS) - 1) & 1)) {
          ok = false;
          break;
        }
        const int key0 = kstart + s * C::SK;
        const int nk = min(C::SK, kend - key0);
        const int nseg = (nk + br - 1) >> br_log2;
        uint32_t bytes = static_cast<uint32_t>(nseg * br * C::ROW_BYTES * 2);
        if constexpr (C::kU8) bytes += static_cast<uint32_t>(nseg * br * 2 * 4);
        uint8_t* st = smem + slot * C::STAGE;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], bytes);
        __syncwarp();
        // one copy per lane: a copy instruction costs its thread hundreds of
        // cycles, so copies issued by one lane in a row would pace the stream
        const int nt = nseg * C::CHUNKS;
        // K: CHUNKS boxes per segment; V: the same, or for u8 one dim-major
        // [head dim][key] box per segment
        const int nv = C::kU8 ? nseg : nt;
        int ncopy = nt + nv;
        if constexpr (C::kU8) ncopy += nseg * (br == a.ps ? 2 : 4);
        for (int c = lane; c < ncopy; c += 32) {
          if (C::kU8 && c >= nt && c < nt + nv) {
            const int seg = c - nt;
            const int key = key0 + (seg << br_log2);
            const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
            const int id = blk[lp - lp0];
            tma_load_4d(st + C::TILE + seg * (D << br_log2), &tmV, slot0, 0, g, id, &full[slot]);
          } else if (c < (C::kU8 ? nt : 2 * nt)) {
            const bool is_v = c >= nt;
            const int j = is_v ? c - nt : c;
            const int seg = j / C::CHUNKS, ch = j % C::CHUNKS;
            const int key = key0 + (seg << br_log2);
            const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
            const int id = blk[lp - lp0];
            const uint32_t off = static_cast<uint32_t>(((seg * C::CHUNKS + ch) << br_log2) * 128);
            tma_load_4d(st + (is_v ? C::TILE : 0) + off, is_v ? &tmV : &tmK, ch * C::ELEMS_128, slot0, g, id,
                        &full[slot]);
            if (!is_v && a.trace != nullptr && ch == 0 && slot0 == 0)
              atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
          } else if constexpr (C::kU8) {
            // per segment [scales(br) | zero-points(br)]; one copy per cache
            // when the segment is a whole page (the record keeps both arrays
            // adjacent), else scales and zero-points separately
            const size_t rec = static_cast<size_t>(a.ps) * (D + 4);
            const int idx = c - nt - nv;
            const bool whole = (br == a.ps);
            const int seg = whole ? idx >> 1 : idx >> 2;
            const bool is_v = whole ? (idx & 1) != 0 : (idx & 2) != 0;
            const int part = whole ? 0 : (idx & 1);  // 0: scales, 1: zero-points
            const int key = key0 + (seg << br_log2);
            const int lp = key >> a.ps_log2, slot0 = key & (a.ps - 1);
            const int id = blk[lp - lp0];
            const size_t roff = (static_cast<size_t>(id) * a.Hkv + g) * rec + static_cast<size_t>(a.ps) * D;
            uint8_t* dst = st + 2 * C::TILE + seg * 4 * br + (is_v ? 4 * C::SK : 0);
            const uint8_t* src = (is_v ? a.v_bytes : a.k_bytes) + roff;
            if (whole) bulk_load(dst, src, 4 * br, &full[slot]);
            else bulk_load(dst + 2 * br * part, src + 2 * a.ps * part + 2 * slot0, 2 * br, &full[slot]);
          }
        }
        issued = s + 1;
      }
      if (!ok) {
        if (lane == 0) {
          atomicOr(a.status, PA_STATUS_TIMEOUT);
          atomicOr(&s_timeout, 1);
        }
        // let the copies already in flight land before the CTA can retire
        for (int s = max(0, issued - C::NS); s < issued; ++s) mbar_wait(&full[s % C::NS], (s / C::NS) & 1);
      }
      return;
    }
  }

  // =========================== consumer warps ==============================
  const int g8 = lane >> 2, tig = lane & 3;
  int RG = (R + RPW - 1) / RPW;
  RG = RG <= 1 ? 1 : (RG <= 2 ? 2 : 4);
  const int KS = kConsumerWarps / RG;
  const int rg = warp % RG, ks = warp / RG;
  const int row_base = rg * RPW;
  const int nvalid = min(max(R - row_base, 0), RPW);
  const int nt_active = (nvalid + 7) >> 3;
  const int L = si.L;

  // Key limits of the rows this thread's accumulator columns hold (rows past
  // R borrow the last valid row's limits so they mask like it).
  // With a tree mask a row may see any new token its mask names: hi covers
  // them all and the mask decides; without one the mask is all ones and hi
  // is the row's own position (the causal chain).
  // (TREE: the launcher picks this instantiation when a mask is given)
  constexpr bool tree = TREE;
  int rlo[NT][2], rhi[NT][2];
  uint32_t rmask[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = min(row_base + nt * 8 + 2 * tig + j, R - 1);
      rhi[nt][j] = tree ? L + si.T - 1 : L + r / a.G;
      rlo[nt][j] = a.window > 0 ? L + r / a.G - a.window + 1 : INT_MIN;
      rmask[nt][j] = tree ? row_new_token_mask(a.tree_mask, si.t0 + r / a.G, r / a.G) : 0xffffffffu;
    }
  const int last_row = row_base + max(nvalid, 1) - 1;
  const int wmin_hi = tree ? L - 1 : L + min(row_base, R - 1) / a.G;
  const int wmax_lo = a.window > 0 ? L + min(last_row, R - 1) / a.G - a.window + 1 : INT_MIN;

  // Q^T fragments (B operand), loaded once.
  uint32_t qf[C::KSTEPS][NT][2];
  float qs[NT][2];  // sum of the row's (f16) query, u8 path only
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = row_base + nt * 8 + g8;
    const bool rv = r < R;
    const int t = si.t0 + (rv ? r / a.G : 0), h = g * a.G + (rv ? r % a.G : 0);
    const size_t qoff = (static_cast<size_t>(t) * a.Hq + h) * D;
    float qsum = 0.f;
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS; ++kk) {
      if constexpr (!C::kU8) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(a.q) + qoff);
        qf[kk][nt][0] = rv ? ld_once(src + (16 * kk + 2 * tig) / 2) : 0u;
        qf[kk][nt][1] = rv ? ld_once(src + (16 * kk + 8 + 2 * tig) / 2) : 0u;
      } else {
        const int dc = kk >> 3, half = (kk >> 2) & 1, sub = kk & 3;
        const int d0 = 128 * dc + 16 * (tig + 4 * half) + 4 * sub;
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          x[e] = rv ? __half2float(__float2half_rn(load_q_elem(a.q, a.q_dtype, qoff + d0 + e))) : 0.f;
        qf[kk][nt][0] = pack2<false>(x[0], x[1]);
        qf[kk][nt][1] = pack2<false>(x[2], x[3]);
        qsum += (x[0] + x[1]) + (x[2] + x[3]);
      }
    }
    if constexpr (C::kU8) {
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
#pragma unroll
      for (int j = 0; j < 2; ++j) qs[nt][j] = __shfl_sync(0xffffffffu, qsum, (2 * tig + j) * 4);
    } else {
      qs[nt][0] = qs[nt][1] = 0.f;
    }
  }

  float m_r[NT][2], l_r[NT][2], zc[NT][2];
  float o[C::MTILES][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      m_r[nt][j] = -INFINITY;
      l_r[nt][j] = 0.f;
      zc[nt][j] = 0.f;
    }
#pragma unroll
  for (int mt = 0; mt < C::MTILES; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;

  // Per-lane ldmatrix roles: K tile (A of S^T, not transposed) and V tile
  // (A of O^T, transposed).
  const int mK = ((lane >> 3) & 1) * 8 + (lane & 7), hiK = (lane >> 4) & 1;
  const int mV = ((lane >> 4) & 1) * 8 + (lane & 7), hiV = (lane >> 3) & 1;
  const float sl2 = a.scale_log2;
  bool timed_out = false;
  // Byte offset of 16-byte unit `unit` of 128-byte column chunk `ch` of the
  // stage's key kk: the TMA's swizzled boxes, or the gather's padded rows.
  auto row_unit = [&](int kk, int ch, int unit) -> uint32_t {
    if constexpr (GATHER) return static_cast<uint32_t>(kk * C::PITCH + ch * 128 + unit * 16);
    else return tile_row_off(kk, ch, a.box_log2, C::CHUNKS) + swz(unit, kk);
  };

  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % C::NS;
    if (!mbar_wait(&full[slot], (s / C::NS) & 1)) {
      timed_out = true;
      break;
    }
    uint8_t* st = smem + slot * C::STAGE;
    const uint32_t kt = smem_u32(st), vt = kt + C::TILE;
    const int key0 = kstart + s * C::SK;
    if (nt_active > 0) {
      // chunks are dealt round-robin over the key-split warps across stages,
      // so short stages (two chunks) still keep every warp busy
      const int c0 = (ks - (s * C::CHUNKS_PER_STAGE) % KS + KS) % KS;
      for (int c = c0; c < C::CHUNKS_PER_STAGE; c += KS) {
        const int ck0 = key0 + 16 * c;
        if (ck0 >= kend) break;
        const int kg0 = ck0 + (C::kU8 ? g8 : key_perm(g8));  // keys of accumulator rows g8 and g8 + 8
        const int kg1 = kg0 + 8;

        // ---------------- S^T = K . Q^T ----------------
        float sa[2][NT][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sa[u][nt][e] = 0.f;
        float ksc[2] = {1.f, 1.f}, kzp[2] = {0.f, 0.f};
        if constexpr (!C::kU8) {
          const int kk = 16 * c + key_perm(mK);
#pragma unroll
          for (int k = 0; k < C::KSTEPS; ++k) {
            const int col = 16 * k;
            const int ch = col / C::ELEMS_128;
            const int unit = ((col % C::ELEMS_128) >> 3) + hiK;
            uint32_t af[4];
            ldsm_x4(kt + row_unit(kk, ch, unit), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt < nt_active) mma16816<kBf>(sa[k & 1][nt], af, qf[k][nt][0], qf[k][nt][1]);
          }
        } else {
          uint4 kw[2][C::CHUNKS][2];
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            const int kk = 16 * c + g8 + 8 * kh;
#pragma unroll
            for (int dc = 0; dc < C::CHUNKS; ++dc)
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                kw[kh][dc][hf] = *reinterpret_cast<const uint4*>(
                    st + tile_row_off(kk, dc, a.box_log2, C::CHUNKS) + swz(tig + 4 * hf, kk));
            const __half* scp = reinterpret_cast<const __half*>(st + 2 * C::TILE + (kk >> a.box_log2) * 4 *
                                                                (1 << a.box_log2));
            const int o = kk & ((1 << a.box_log2) - 1);
            ksc[kh] = __half2float(scp[o]) * sl2;
            kzp[kh] = __half2float(scp[(1 << a.box_log2) + o]);
          }
#pragma unroll
          for (int k = 0; k < C::KSTEPS; ++k) {
            const int dc = k >> 3, hf = (k >> 2) & 1, sub = k & 3;
            const uint32_t w0 = reinterpret_cast<const uint32_t*>(&kw[0][dc][hf])[sub];
            const uint32_t w1 = reinterpret_cast<const uint32_t*>(&kw[1][dc][hf])[sub];
            uint32_t af[4];
            af[0] = u8pair_to_f16x2(w0, 0x4140u);
            af[1] = u8pair_to_f16x2(w1, 0x4140u);
            af[2] = u8pair_to_f16x2(w0, 0x4342u);
            af[3] = u8pair_to_f16x2(w1, 0x4342u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt < nt_active) mma16816<false>(sa[k & 1][nt], af, qf[k][nt][0], qf[k][nt][1]);
          }
        }

        // ---------------- scale, mask, online softmax ----------------
        const bool clean = ck0 >= wmax_lo && ck0 + 15 <= wmin_hi;
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float acc = sa[0][nt][e] + sa[1][nt][e];
            float v;
            if constexpr (C::kU8) v = (acc - kzp[e >> 1] * qs[nt][e & 1]) * ksc[e >> 1];
            else v = acc * sl2;
            if (!clean) {
              const int key = (e >> 1) ? kg1 : kg0;
              bool okk = key >= rlo[nt][e & 1] && key <= rhi[nt][e & 1];
              if constexpr (TREE) okk = okk && (key < L || ((rmask[nt][e & 1] >> (key - L)) & 1u));
              v = okk ? v : -INFINITY;
            }
            sc[nt][e] = v;
          }
        float alpha[NT][2];
        bool need_rescale = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sc[nt][j], sc[nt][2 + j]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(m_r[nt][j], mx);
            const float mu = (mnew == -INFINITY) ? 0.f : mnew;
            alpha[nt][j] = ex2(m_r[nt][j] - mu);
            need_rescale |= (mnew != m_r[nt][j]);
            m_r[nt][j] = mnew;
            sc[nt][j] = ex2(sc[nt][j] - mu);
            sc[nt][2 + j] = ex2(sc[nt][2 + j] - mu);
            l_r[nt][j] = l_r[nt][j] * alpha[nt][j] + sc[nt][j] + sc[nt][2 + j];
          }
        if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll
          for (int mt = 0; mt < C::MTILES; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) o[mt][nt][e] *= alpha[nt][e & 1];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) zc[nt][j] *= alpha[nt][j];
        }

        // ---------------- P^T (B operand of O^T = V^T P^T) ----------------
        uint32_t pb[NT][2];
        if constexpr (!C::kU8) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movmatrix_t(pack2<kBf>(sc[nt][0], sc[nt][1]));
            pb[nt][1] = movmatrix_t(pack2<kBf>(sc[nt][2], sc[nt][3]));
          }
        } else {
          float vsc[2], vzp[2];
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            const int kk = 16 * c + g8 + 8 * kh;
            const int key = kk + key0;
            const bool in_union = key >= si.klo && key <= si.khi;
            const __half* scp = reinterpret_cast<const __half*>(st + 2 * C::TILE + 4 * C::SK +
                                                                (kk >> a.box_log2) * 4 * (1 << a.box_log2));
            const int o = kk & ((1 << a.box_log2) - 1);
            vsc[kh] = in_union ? __half2float(scp[o]) : 0.f;
            vzp[kh] = in_union ? __half2float(scp[(1 << a.box_log2) + o]) : 0.f;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint32_t h0 = pack2<false>(sc[nt][0] * vsc[0], sc[nt][1] * vsc[0]);
            const uint32_t h1 = pack2<false>(sc[nt][2] * vsc[1], sc[nt][3] * vsc[1]);
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
            zc[nt][0] += f0.x * vzp[0] + f1.x * vzp[1];
            zc[nt][1] += f0.y * vzp[0] + f1.y * vzp[1];
            pb[nt][0] = movmatrix_t(h0);
            pb[nt][1] = movmatrix_t(h1);
          }
        }

        // ---------------- O^T += V^T . P^T ----------------
        if constexpr (!C::kU8) {
          if (ck0 < si.klo || ck0 + 15 > si.khi) {
            // keys outside every row's range may hold garbage (even NaN);
            // their weight is 0, but 0 * NaN is not, so clear those V rows.
            constexpr int UNITS = C::ROW_BYTES / 16;
            for (int idx = lane; idx < 16 * UNITS; idx += 32) {
              const int m = idx / UNITS, u = idx % UNITS;
              const int key = ck0 + m;
              if (key < si.klo || key > si.khi)
                *reinterpret_cast<uint4*>(st + C::TILE + (GATHER ? (16 * c + m) * C::PITCH + 16 * u
                                                                 : tile_row_off(16 * c + m, u >> 3, a.box_log2,
                                                                                C::CHUNKS) + 16 * (u & 7))) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async();
            __syncwarp();
          }
          const int kk = 16 * c + key_perm(mV);
#pragma unroll
          for (int mt = 0; mt < C::MTILES; ++mt) {
            const int col = 16 * mt;
            const int ch = col / C::ELEMS_128;
            const int unit = ((col % C::ELEMS_128) >> 3) + hiV;
            uint32_t af[4];
            ldsm_x4_t(vt + row_unit(kk, ch, unit), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt < nt_active) mma16816<kBf>(o[mt][nt], af, pb[nt][0], pb[nt][1]);
          }
        } else {
          // A = V^T (16 head dims x 16 keys) straight from the dim-major
          // tile [segment][head dim][key]: thread (g8, tig) takes keys
          // 2tig, 2tig+1 (and + 8) of head dims 16mt + g8 (and + 8), two
          // adjacent codes per 16-bit load
          const int brl = a.box_log2;
          const uint8_t* vt8 = st + C::TILE;
          const int k0 = 16 * c + 2 * tig, k1 = k0 + 8;
          const int off0 = ((k0 >> brl) * D) << brl | (k0 & ((1 << brl) - 1));
          const int off1 = ((k1 >> brl) * D) << brl | (k1 & ((1 << brl) - 1));
          const __half2 k1024 = __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
#pragma unroll
          for (int mt = 0; mt < C::MTILES; ++mt) {
            const int d0 = 16 * mt + g8;
            uint32_t af[4];
            const uint32_t c00 = *reinterpret_cast<const uint16_t*>(vt8 + off0 + (d0 << brl));
            const uint32_t c10 = *reinterpret_cast<const uint16_t*>(vt8 + off0 + ((d0 + 8) << brl));
            const uint32_t c01 = *reinterpret_cast<const uint16_t*>(vt8 + off1 + (d0 << brl));
            const uint32_t c11 = *reinterpret_cast<const uint16_t*>(vt8 + off1 + ((d0 + 8) << brl));
            const uint32_t w[4] = {c00, c10, c01, c11};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t h = __byte_perm(w[i], 0x64646464u, 0x4140u);
              const __half2 cv = __hsub2(*reinterpret_cast<const __half2*>(&h), k1024);
              af[i] = *reinterpret_cast<const uint32_t*>(&cv);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt < nt_active) mma16816<false>(o[mt][nt], af, pb[nt][0], pb[nt][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (timed_out && lane == 0) {
    atomicOr(a.status, PA_STATUS_TIMEOUT);
    atomicOr(&s_timeout, 1);
  }

  // =========================== merge & write ===============================
  consumer_sync();  // every consumer is done with the stage ring
  if (s_bad) {
    // corrupt block table: poison this partition (the combine zeroes the rows)
    for (int idx = threadIdx.x; idx < R * D; idx += kConsumerWarps * 32) {
      const int r = idx / D, d = idx % D;
      const size_t row = static_cast<size_t>(si.t0 + r / a.G) * a.Hq + g * a.G + r % a.G;
      if (si.nparts == 1) {
        store_out(a.out, a.out_dtype, row * D + d, 0.f);
      } else if (d == 0) {
        a.pm[prow(row, si, a.Hq) * a.num_parts + p] = 0.f;
        a.pl[prow(row, si, a.Hq) * a.num_parts + p] = -1.f;
      }
    }
    return;
  }
  float* mo = reinterpret_cast<float*>(smem);
  float* mm = mo + kConsumerWarps * RPW * S::MERGE_LD;
  float* ml = mm + kConsumerWarps * RPW;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = l_r[nt][j], z = zc[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      z += __shfl_xor_sync(0xffffffffu, z, 4);
      z += __shfl_xor_sync(0xffffffffu, z, 8);
      z += __shfl_xor_sync(0xffffffffu, z, 16);
      l_r[nt][j] = l;
      zc[nt][j] = z;
      if (g8 == 0) {
        mm[warp * RPW + nt * 8 + 2 * tig + j] = m_r[nt][j];
        ml[warp * RPW + nt * 8 + 2 * tig + j] = l;
      }
    }
#pragma unroll
  for (int mt = 0; mt < C::MTILES; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rl = nt * 8 + 2 * tig + (e & 1);
        const int d = out_dim<D, C::kU8>(mt, g8 + 8 * (e >> 1));
        mo[(warp * RPW + rl) * S::MERGE_LD + d] = o[mt][nt][e] - zc[nt][e & 1];
      }
  consumer_sync();

  const bool poisoned = s_timeout != 0;
  // One warp per row: the row's key-split weights and its output offset once
  // (no per-element index arithmetic), then four head dims per lane.
  for (int r = warp; r < R; r += kConsumerWarps) {
    const int rgr = r / RPW, rl = r % RPW;
    float M = -INFINITY;
    for (int k2 = 0; k2 < KS; ++k2) M = fmaxf(M, mm[(k2 * RG + rgr) * RPW + rl]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float wgt[kConsumerWarps];
    float lsum = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < kConsumerWarps; ++k2) {
      wgt[k2] = 0.f;
      if (k2 < KS) {
        const int wr = (k2 * RG + rgr) * RPW + rl;
        wgt[k2] = ex2(mm[wr] - Mu);
        lsum += wgt[k2] * ml[wr];
      }
    }
    const int tq = r / a.G;
    const size_t row = static_cast<size_t>(si.t0 + tq) * a.Hq + g * a.G + (r - tq * a.G);
    const float inv = (poisoned || !(lsum > 0.f)) ? 0.f : 1.f / lsum;
    const size_t pr = prow(row, si, a.Hq) * a.num_parts + p;
    for (int d = 4 * lane; d < D; d += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k2 = 0; k2 < kConsumerWarps; ++k2) {
        if (k2 < KS) {
          const float4 x = *reinterpret_cast<const float4*>(mo + ((k2 * RG + rgr) * RPW + rl) * S::MERGE_LD + d);
          acc.x = fmaf(wgt[k2], x.x, acc.x);
          acc.y = fmaf(wgt[k2], x.y, acc.y);
          acc.z = fmaf(wgt[k2], x.z, acc.z);
          acc.w = fmaf(wgt[k2], x.w, acc.w);
        }
      }
      if (si.nparts == 1)
        store_out4(a.out, a.out_dtype, row * D + d,
                   poisoned ? make_float4(0.f, 0.f, 0.f, 0.f)
                            : make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
      else
        *reinterpret_cast<float4*>(a.po + pr * D + d) = acc;
    }
    if (si.nparts > 1 && lane == 0) {
      a.pm[pr] = M;
      a.pl[pr] = poisoned ? -1.f : lsum;
    }
  }
}

}  // namespace pa
