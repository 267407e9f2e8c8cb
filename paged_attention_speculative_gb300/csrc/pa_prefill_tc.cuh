// pa_prefill_tc.cuh — prefill chunks of a mixed batch on the 5th-generation
// tensor cores: sequences with more than 8 new tokens (a chunk of a prompt
// beside the verify steps of other sequences, the MIXED stage of the OpenVINO
// paged-attention op that issue 38153 describes).
//
// One CTA per (row block, KV head).  A row block is 128 or 256 query rows
// (the launcher's choice): TQ = rows / G consecutive new tokens of one
// sequence times the G query heads
// of the KV head, ordered like the verify kernels' rows (r -> token r / G,
// head g * G + r % G), split into two 128-row tiles that share every K/V
// stage.  The CTA streams its keys [klo, khi] once, klo the window start of
// its first token and khi = past_len + its last token:
//   S_t(s) = Q_t . K_s^T   tcgen05.mma M=128, N=64, K=D  (Q_t from smem)
//   P_t(s) = 2^(S*scale*log2e - m) per row, causal / window mask per row
//   O_t   += P_t(s) . V_s  tcgen05.mma M=128, N=D, K=64  (P_t in TMEM)
// and writes the normalised rows directly -- or, when the blocks' keys are
// split (chunks whose blocks fill at most half the SMs: as many pieces as
// still fit in one wave, up to grid.z), each CTA streams one contiguous run
// of the block's stages and writes unnormalised partial rows (max,
// denominator, output) that pa_prefill_combine merges, as the verify path's
// combine does.
//
// With two tiles they ping-pong, one S and one P buffer each: the MMA thread
// issues S_0(s), PV_1(s-1), S_1(s), PV_0(s), so tile 0's softmax of stage s
// runs while tile 1's scores are computed, and tile 1's while tile 0's next
// scores are; each SM sub-partition holds one softmax warp of each tile.
// With one tile (blocks of 128 rows), tile 0 uses both tiles' S and P
// columns as two buffers and S(s+1) is issued before PV(s).
//
// Warp roles (320 threads):
//   warps 0-3  softmax of tile 0: thread owns row (warp % 4) * 32 + lane (TMEM lane)
//   warps 4-7  softmax of tile 1 (idle when the block has 128 rows or fewer)
//   warp 8     MMA issuer (one thread)
//   warp 9     TMA producer: block ids one stage ahead, one tile load per
//              page segment and 128-byte chunk
// Row blocks are numbered over the batch's prefill sequences in order, each
// sequence's blocks last token first (the longest start first); each CTA
// finds its (sequence, first token) by walking subsequence_begins.
#pragma once

#include "pa_partition_tc.cuh"

namespace pa {

template <int D, int KV>
struct PfCfg {
  static_assert(KV == KV_BF16 || KV == KV_F16, "prefill tiles take 16-bit caches");
  static_assert(D == 64 || D == 128, "prefill tiles: head_dim 64 or 128");
  static constexpr bool kBf16 = (KV == KV_BF16);
  static constexpr int SK = 64;                  // keys per stage
  static constexpr int CH = D / 64;              // 128-byte chunks per row
  static constexpr int TILE = SK * D * 2;        // one K (or V) stage tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int QT = 128 * D * 2;         // one query tile, [chunk][row][128 B]
  static constexpr int RING_OFF = 2 * QT;
  static constexpr int FIXED = 2 * QT + 512 + 1024;
  static constexpr int NS_FIT = (226 * 1024 - FIXED) / STAGE;
  static constexpr int NS = NS_FIT > 8 ? 8 : NS_FIT;
  static constexpr int BAR_OFF = RING_OFF + NS * STAGE;
  static constexpr int BYTES = BAR_OFF + 512 + 1024;
  // TMEM columns: O_t [t D, t D + D), S_t [2 D + t SK, +SK), P_t (16-bit
  // pairs) [2 D + 2 SK + t SK / 2, +SK / 2)
  static constexpr int S_COL = 2 * D;
  static constexpr int P_COL = 2 * D + 2 * SK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = tc_idesc(128, SK, kBf16, false);
  static constexpr uint32_t IDESC_PV = tc_idesc(128, D, kBf16, true);
  static_assert(NS >= 3, "pipeline needs a few stages");
  static_assert(P_COL + SK <= TMEM_COLS, "tensor-memory budget");
};

// SPLIT: the launch may split the blocks' keys into pieces (grid.z > 1); the
// instantiation without it keeps the unsplit kernel's code exactly.
template <int D, int KV, bool SPLIT>
__global__ void __launch_bounds__(320, 1)
    pa_prefill_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const PartArgs a) {
  using C = PfCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::RING_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* full = bars;                 // [NS] TMA landed
  uint64_t* empty = full + C::NS;        // [NS] stage consumed (MMA commit after the last PV)
  uint64_t* s_full = empty + C::NS;      // [2] S_t written (MMA commit)
  uint64_t* s_free = s_full + 2;         // [2] S_t read (4 softmax warps of tile t)
  uint64_t* p_full = s_free + 2;         // [2] P_t written (4 softmax warps of tile t)
  uint64_t* pv_done = p_full + 2;        // [2] PV_t done (MMA commit)
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout, s_pieces;

  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int TQ = a.row_cap / a.G;  // new tokens per row block (a.row_cap = 128 or 256 rows)
  pdl_wait_primary();        // inputs and outputs may belong to the previous kernel

  // ---- which sequence and tokens this row block covers ----
  int b = -1, i0 = 0;
  {
    long long blk = blockIdx.x;
    for (int s = 0; s < a.num_seqs; ++s) {
      const int T = ld_once(a.begins + s + 1) - ld_once(a.begins + s);
      if (T <= PA_MAX_QUERY_LEN) continue;  // a verify step (or malformed: reported below)
      const long long nb = (T + TQ - 1) / TQ;
      if (blk < nb) {
        b = s;
        i0 = static_cast<int>(nb - 1 - blk) * TQ;  // last tokens (most keys) first
        break;
      }
      blk -= nb;
    }
  }
  // pieces in use: the launch's grid.z is an upper bound made on the host,
  // which does not know the chunks' lengths
  int npieces = 1;
  if constexpr (SPLIT) npieces = prefill_pieces(a.begins, a.num_seqs, TQ, a.Hkv, gridDim.z, a.num_sms);
  pdl_launch_dependents();
  if (b < 0 || (SPLIT && static_cast<int>(blockIdx.z) >= npieces)) return;
  const SeqInfo si = seq_info(a.begins, a.past_lens, b, a.total_tokens, a.G, a.ps, a.max_ctx, a.window,
                              a.part_tokens, a.row_cap, kRoleLong);
  const int ntok = min(TQ, si.T - i0);  // tokens of this row block
  const int R = ntok * a.G;             // real rows (at most 256)
  if (si.err) {
    if (threadIdx.x == 0) atomicOr(a.status, si.err);
    if (si.rows_ok && (!SPLIT || blockIdx.z == 0))
      for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        store_out(a.out, a.out_dtype, (static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G) * D + d,
                  0.f);
      }
    return;
  }
  if (ntok <= 0) return;
  const bool two = R > 128;  // block-uniform: tile 1 has real rows

  const int klo = a.window > 0 ? max(0, si.L + i0 - a.window + 1) : 0;
  const int khi = si.L + i0 + ntok - 1;
  const int kfirst = (klo >> a.ps_log2) << a.ps_log2;  // page aligned
  // piece blockIdx.z of this block's `pieces` streams its stages [st0, st1)
  const int pieces = SPLIT ? prefill_block_pieces(npieces, khi + 1 - kfirst) : 1;
  if (SPLIT && static_cast<int>(blockIdx.z) >= pieces) return;
  const int n_all = (khi + 1 - kfirst + C::SK - 1) / C::SK;
  const int st0 = SPLIT ? static_cast<int>(static_cast<long long>(n_all) * blockIdx.z / pieces) : 0;
  const int st1 = SPLIT ? static_cast<int>(static_cast<long long>(n_all) * (blockIdx.z + 1) / pieces) : n_all;
  const int kstart = kfirst + st0 * C::SK;             // this piece's first key
  const int kend = SPLIT ? min(kfirst + st1 * C::SK, khi + 1) : khi + 1;  // one past its last
  const int n_stages = st1 - st0;

  if (threadIdx.x == 288) {
    s_bad = 0;
    s_timeout = 0;
    if constexpr (SPLIT) s_pieces = pieces;  // read back by the epilogue (no register held over the loop)
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], two ? 1 : 2);  // one producer, or K and V producers (one tile)
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 4);
      mbar_init(&p_full[t], 4);
      mbar_init(&pv_done[t], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t tmem = 0;
  if (warp < 9) {
    if (warp == 0) {
      tmem_alloc(&s_tmem, C::TMEM_COLS);
      tmem_relinquish();
    }
    if (warp < 8) {
      // Q rows into shared memory, 128B-swizzled K-major tiles (the layout a
      // TMA load would give): unit u of row rr of tile t at
      // t QT + (c 128 + rr) 128 + (u ^ (rr & 7)) 16; rows past the block's
      // tokens are zero
      const int r = warp * 32 + lane, t = r >> 7, rr = r & 127;
      const bool real = r < R;
      const size_t row = real ? static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + row * D);
#pragma unroll
      for (int c = 0; c < C::CH; ++c)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = real ? __ldg(src + 8 * c + u) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(smem + t * C::QT + (c * 128 + rr) * 128 + ((u ^ (rr & 7)) << 4)) = x;
        }
      fence_proxy_async();  // Q, seen by the tensor cores' proxy
    }
    tc_fence_before();
    bar_sync_n(2, 288);  // the TMEM address is published and Q is in place
    tc_fence_after();
    tmem = s_tmem;
  }

  // MMA issue steps (one thread each: warp 8, and warp 4 for PV with one tile)
  // S of tile t for stage s into score buffer bi
  auto issue_s = [&](int t, int bi, int s) {
    const uint32_t k_base = smem_u32(ring + (s % C::NS) * C::STAGE);
    const uint32_t q_base = smem_u32(smem + t * C::QT);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c = kk >> 2, w = kk & 3;
      const uint64_t ad = sw128_desc(q_base + c * 128 * 128 + 32 * w, 16, 1024);
      const uint64_t bd = sw128_desc(k_base + c * C::SK * 128 + 32 * w, 16, 1024);
      tc_mma(tmem + C::S_COL + bi * C::SK, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
    }
    tc_commit(&s_full[bi]);
  };
  // O_t += P (buffer bi, written in phase ph) . V_s
  auto issue_pv = [&](int t, int bi, uint32_t ph, int s) -> bool {
    if (!mbar_wait(&p_full[bi], ph)) return false;
    tc_fence_after();
    const uint32_t v_base = smem_u32(ring + (s % C::NS) * C::STAGE + C::TILE);
#pragma unroll
    for (int j = 0; j < C::SK / 16; ++j) {
      const uint64_t bd = sw128_desc(v_base + j * 16 * 128, C::SK * 128, 1024);
      tc_mma_ta(tmem + t * D, tmem + C::P_COL + bi * (C::SK / 2) + 8 * j, bd, C::IDESC_PV,
                (s > 0 || j > 0) ? 1u : 0u);
    }
    tc_commit(&pv_done[bi]);
    return true;
  };

  // The stage ring's copies: K and V tiles of each page segment, one
  // (segment, chunk) pair per lane.  With two tiles warp 9 issues both; with
  // one, warp 9 issues K and the idle warp 5 V -- a copy instruction costs
  // its warp hundreds of cycles, and one producer paced the ring.
  auto produce = [&](bool do_k, bool do_v) {
    const int32_t* bt = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
    const int br_log2 = a.box_log2, br = 1 << br_log2;  // rows per tile load (page size, at most 64)
    int bad = 0;
    // block id of segment `lane` of stage s (0 past the block's keys)
    auto load_id = [&](int s) -> int {
      const int key = kstart + s * C::SK + (lane << br_log2);
      return (lane < (C::SK >> br_log2) && key < kend) ? __ldg(bt + (key >> a.ps_log2)) : 0;
    };
    const int parts = (do_k ? 1 : 0) + (do_v ? 1 : 0);
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
      uint8_t* st = ring + slot * C::STAGE;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(parts * nseg * br * D * 2));
      __syncwarp();
      const int seg = lane / C::CH, c = lane % C::CH;  // one (segment, chunk) pair per lane: nseg * CH <= 16
      const int sid = __shfl_sync(0xffffffffu, id, seg & 31);
      if (lane < nseg * C::CH) {
        const int key = key0 + (seg << br_log2);
        const uint32_t off = static_cast<uint32_t>((c * C::SK + (seg << br_log2)) * 128);
        if (do_k) tma_load_4d(st + off, &tmK, c * 64, key & (a.ps - 1), g, sid, &full[slot]);
        if (do_v) tma_load_4d(st + C::TILE + off, &tmV, c * 64, key & (a.ps - 1), g, sid, &full[slot]);
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      s_bad = 1;
      atomicOr(a.status, PA_STATUS_BLOCK_ID);
    }
  };

  if (warp == 9) {
    // =========================== TMA producer ===============================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    produce(true, two);
  } else if (warp == 5 && !two) {
    // ===================== V producer (one tile) ============================
    produce(false, true);
  } else if (warp == 8) {
    // =========================== MMA issuer =================================
    // Per stage s: S_0(s); [PV_1(s-1); S_1(s)]; PV_0(s).  A stage's slot is
    // released after the last PV that reads it.
    if (lane == 0) {
      bool ok = true;
      if (two) {
        // two tiles, one buffer each (index t, phase s & 1):
        // S_0(s); PV_1(s-1); S_1(s); PV_0(s)
        for (int s = 0; s < n_stages && ok; ++s) {
          if (!mbar_wait(&full[s % C::NS], (s / C::NS) & 1) || (s >= 1 && !mbar_wait(&s_free[0], (s - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(0, 0, s);
          if (s >= 1) {
            if (!(ok = issue_pv(1, 1, (s - 1) & 1, s - 1))) break;
            tc_commit(&empty[(s - 1) % C::NS]);
            if (!mbar_wait(&s_free[1], (s - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          issue_s(1, 1, s);
          if (!(ok = issue_pv(0, 0, s & 1, s))) break;
        }
        if (ok && n_stages >= 1) {
          ok = issue_pv(1, 1, (n_stages - 1) & 1, n_stages - 1);
          if (ok) tc_commit(&empty[(n_stages - 1) % C::NS]);
        }
      } else {
        // one tile, two buffers (index s & 1, phase (s >> 1) & 1): this
        // thread issues the scores only, as soon as the stage has landed
        // and its buffer is read; warp 4 issues the PVs, so a score MMA
        // never waits behind a PV for the softmax
        for (int s = 0; s < n_stages && ok; ++s) {
          const int sb = s & 1;
          if (!mbar_wait(&full[s % C::NS], (s / C::NS) & 1) ||
              (s >= 2 && !mbar_wait(&s_free[sb], ((s >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(0, sb, s);
        }
      }
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else if (warp == 4 && !two) {
    // ===================== PV issuer (one tile) =============================
    if (lane == 0) {
      bool ok = true;
      for (int s = 0; s < n_stages && ok; ++s) {
        ok = issue_pv(0, s & 1, (s >> 1) & 1, s);
        if (ok) tc_commit(&empty[s % C::NS]);  // its score MMA finished before the softmax began
      }
      if (!ok) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else if (warp < 4 || two) {
    // ===================== softmax warps of tile t (rows) ===================
    const int t = warp >> 2, quarter = warp & 3;
    const int r = t * 128 + quarter * 32 + lane;  // row of the block (TMEM lane r % 128 of tile t)
    const int rc = min(r, R - 1);                 // padding rows mask like the last real row
    const int i = i0 + rc / a.G;                  // the row's new token
    const int hi = si.L + i;
    const int lo = a.window > 0 ? si.L + i - a.window + 1 : INT_MIN;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tm_o = tmem + t * D + lane_off;
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int s = 0; s < n_stages; ++s) {
      // buffer and barrier index of this stage's S and P, and the phase of
      // stage s on them: one per tile (two tiles), or alternating (one tile)
      const int bi = two ? t : (s & 1);
      const uint32_t ph = two ? (s & 1) : ((s >> 1) & 1);
      if (!mbar_wait(&s_full[bi], ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[C::SK];  // raw scores q.k (the scale is applied inside the exponent)
      tmem_ld64(tmem + C::S_COL + bi * C::SK + lane_off, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[bi]);

      const int key0 = kstart + s * C::SK;
      const bool clean = key0 >= lo && key0 + C::SK - 1 <= hi;
      if (!clean) {
#pragma unroll
        for (int j = 0; j < C::SK; ++j) {
          const int key = key0 + j;
          x[j] = (key >= lo && key <= hi) ? x[j] : -INFINITY;
        }
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
      // O_t is rescaled once PV(s-1) is done; with one P buffer per tile
      // that is also when P(s) may replace P(s-1)
      if (s >= 1 && (two || __any_sync(0xffffffffu, need))) {
        const int pb = two ? t : ((s - 1) & 1);
        const uint32_t pph = two ? ((s - 1) & 1) : (((s - 1) >> 1) & 1);
        if (!mbar_wait(&pv_done[pb], pph)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tm_o + 32 * c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tm_o + 32 * c, o);
          }
        }
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
      // one tile: P buffer s & 1 is free once PV(s-2) is done
      if (!two && s >= 2) {
        if (!mbar_wait(&pv_done[bi], ((s >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tmem + C::P_COL + bi * (C::SK / 2) + lane_off, reinterpret_cast<const float*>(pk));
      // V rows of keys outside the block's range may hold garbage (even NaN):
      // their weights are 0 but 0 * NaN is not, so tile 0's warps clear them
      // (both tiles' PV of the stage are issued after tile 0's P)
      if (t == 0 && (key0 < klo || key0 + C::SK - 1 > khi)) {
        uint8_t* vt = ring + (s % C::NS) * C::STAGE + C::TILE;
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
      if (lane == 0) mbar_arrive(&p_full[bi]);
    }
    // ---- epilogue: normalised O row from TMEM -> output (or the piece's
    // partial row) ----
    if (ok && n_stages >= 1) {
      const int n1 = n_stages - 1;
      if (!mbar_wait(&pv_done[two ? t : (n1 & 1)], two ? (n1 & 1) : ((n1 >> 1) & 1))) ok = false;
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
    tc_fence_after();
    const bool poisoned = s_bad != 0 || s_timeout != 0 || !ok;
    const bool real = r < R;
    const size_t row = real ? static_cast<size_t>(si.t0 + i0 + r / a.G) * a.Hq + g * a.G + r % a.G : 0;
    if (SPLIT && s_pieces > 1) {
      // partial row of this piece (stride: the launch's grid.z); a piece
      // without stages holds nothing (its accumulator was never written) and
      // gets weight 0
      const size_t pr = row * gridDim.z + blockIdx.z;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tm_o + 32 * c, o);
        if (real) {
          float4* dst = reinterpret_cast<float4*>(a.po + pr * D + 32 * c);
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            dst[e / 4] = n_stages > 0 ? make_float4(o[e], o[e + 1], o[e + 2], o[e + 3])
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (real) {
        a.pm[pr] = n_stages > 0 ? m_ref : -INFINITY;
        a.pl[pr] = poisoned ? -1.f : (n_stages > 0 ? l : 0.f);
      }
    } else {
      const float inv = (poisoned || !(l > 0.f)) ? 0.f : 1.f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tm_o + 32 * c, o);
        if (real) {
#pragma unroll
          for (int e = 0; e < 32; ++e) store_out(a.out, a.out_dtype, row * D + 32 * c + e, poisoned ? 0.f : o[e] * inv);
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
