// pa_partition_u8.cuh — split-KV partition kernel for u8 KV caches with a
// per-token fp16 scale and zero-point (OpenVINO issue 38153, reproduction
// step 1: "u8 KV cache precision"), head_dim 128, pages of 16, 32 or 64
// tokens, up to 32 query rows per KV head, on the 5th-generation tensor cores
// with the keys of a stage on the MMA's M dimension.
//
// Same contract as the other partition kernels: one CTA per (partition, KV
// head, sequence); every page of the partition is read once for all T_b x G
// query rows (the GQA read-once of issue 38153, "Cause"); per-token partials,
// or the output when one partition covers the sequence.
//
// The issue's page reports the u8 path as the one whose cost grows fastest
// with the number of query tokens: an ALU-bound dequantisation per element
// and per query row.  Here each code is converted once per stage, whatever the
// row count, by four converter warps that write f16 into tensor memory; the
// per-token scale and zero-point are scalars of the softmax thread that owns
// the key (value = (code - zp) * scale):
//   S^T[k][n] = C'_k . q_n                C'_k = 1024 + K codes of key k (f16, exact)
//   s[k][n]   = ks_k * (S^T[k][n] - (kz_k + 1024) * sum_d q_n)
//   P'[k][n]  = f16(2^(s scale log2e - m_n) * vs_k)
//   O^T[d][n] += sum_k Vc[k][d] P'[k][n]  Vc = V codes (f16, exact)
//   out[n][d] = (O^T[d][n] - sum_k P'[k][n] vz_k) / sum_k 2^(...)
// The +1024 of the K operand (a code's byte placed under the exponent of
// 1024.0) is folded into the zero-point term, so a K code costs one byte
// permute; the V codes are converted exactly because the value correction is
// subtracted from the accumulated sum.  The correction uses the same rounded
// P' that the tensor cores multiply.
//
// Per 128-key stage: the K and V records (codes, scales, zero-points) of the
// stage's pages land in one shared-memory slot with one copy per record — a
// TMA box with 64-byte swizzle for K (so the converters read key rows without
// bank conflicts) and a 1-D bulk copy for V — K and V each under their own
// mbarrier; a ring of NS = 4 such slots keeps ~135 KB in flight per SM.
// Converted codes live in tensor memory in two rings: K buffers (free once
// their S^T MMA is done) and deeper V^T buffers (free only after the PV
// MMA, which follows the softmax).
//
// Warp roles (640 threads, 20 warps; for warps 0-15, q = warp % 4 is the
// TMEM lane quarter a warp may access and h = warp / 8 its half):
//   warps 0-3, 8-11   softmax: half h takes the stages s with s % 2 == h;
//                     thread = key 32q + lane of the stage (TMEM lane of
//                     S^T), all N rows, the half's own running maxima and
//                     O^T accumulator (merged in the epilogue); head dim
//                     32q + lane of O^T in the epilogue; they also stage Q.
//                     A half's four warps share its maxima and rescale
//                     decisions (named barrier 3 + h).
//   warps 4-7, 12-15  converters: thread t = 32q + lane turns head dims
//                     [64h, 64h + 64) of key t's K codes into f16 in TMEM (A
//                     operand of S^T), turns head dim t of keys [64h,
//                     64h + 64) of the V codes (stored dim-major) into TMEM
//                     (A operand of O^T = V^T P'^T), and writes key t's K
//                     (h = 0) or V (h = 1)
//                     scale / zero-point terms (zero for keys out of range).
//   warp 16           K producer: block ids, then per stage one TMA copy
//                     instruction (K records, one lane each); the first NS
//                     stages go out as soon as their ids are read and
//                     checked, while Q is staged
//   warp 19           V producer: per stage one bulk copy instruction (V
//                     records, one lane each).  A copy instruction costs its
//                     warp ~500 cycles whatever the lanes, so K and V are
//                     issued by two warps in parallel, each under its own
//                     mbarrier (the converters start on K before V lands).
//   warp 17           S^T MMA issuer (one thread): S^T(s) once stage s is
//                     converted and its S^T buffer free
//   warp 18           PV MMA issuer (one thread): PV(s) once P'(s) is written
// The compute warps only compute: every copy, MMA issue and the waits they
// need sit on the three control warps.  Two MMA issuers, because a
// tcgen05.mma of these shapes costs its issuing thread ~75-100 cycles and a
// 128-key stage takes 16 of them.
#pragma once

#include "pa_tcgen05.cuh"

namespace pa {

template <int N, int PS>
struct U8Cfg {
  static_assert(N == 16 || N == 32, "row tile 16 / 32");
  static_assert(PS == 16 || PS == 32 || PS == 64, "page size 16 / 32 / 64");
  static constexpr int D = 128;
  static constexpr int SK = 128;                       // keys per stage (M of the score MMA)
  static constexpr int PPS = SK / PS;                  // pages per stage
  static constexpr int REC = PS * (D + 4);             // one page-head record: codes, scales, zero-points
  // K records start on 128-byte boundaries (a swizzled TMA destination); the
  // 64-byte swizzle permutes by absolute shared-memory address bits, and the
  // stages start on 512-byte boundaries (the pattern's period), so a
  // record's bytes sit at sw64(offset in the stage)
  static constexpr int K_SLOT = (REC + 127) / 128 * 128;
  static constexpr int K_AREA = PPS * K_SLOT;
  static constexpr int STAGE = (K_AREA + PPS * REC + 511) / 512 * 512;
  // Converted stages in tensor memory: a K buffer is free once its S^T MMA
  // is done, a V^T buffer only once its PV MMA is (after the softmax), so
  // the V ring is the deeper one.  Stage s + NBV's V conversion waits for
  // PV(s); with a stage's path from landing to PV done ~5,500 cycles, four V
  // buffers keep that wait off the ~1,500-cycle stage period.
  static constexpr int NBK = 2;
  static constexpr int NBV = 4;
  static constexpr int SIDE = SK * 16;                 // float4 per key: ks * scale * log2e, kz + 1024, vs, vz
  static constexpr int Q_BYTES = N * D * 2;            // Q tile (f16), K-major: [chunk][row][128 B]
  static constexpr int P_BYTES = SK * 128;             // P'^T tile (f16), MN-major: [key][64 row slots x 2 B]
  static constexpr int MISC = 7680;
  static constexpr int FIXED = NBV * SIDE + Q_BYTES + 2 * P_BYTES + 4 * kMaxPagesPerCta + MISC + 1024;
  static constexpr int NS_FIT = (226 * 1024 - FIXED) / STAGE;
  // stages in the ring; a fifth stage measured slower (every CTA's first
  // stage then shares HBM with more bytes at start-up) and no faster after
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static constexpr int P_OFF = 0;                      // the 128-byte-swizzled tiles first (1024-aligned)
  static constexpr int Q_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int ST_OFF = Q_OFF + Q_BYTES;       // the ring of stages
  static constexpr int SIDE_OFF = ST_OFF + NS * STAGE;
  static constexpr int BLK_OFF = SIDE_OFF + NBV * SIDE;
  static constexpr int MISC_OFF = BLK_OFF + 4 * kMaxPagesPerCta;
  static constexpr int BYTES = MISC_OFF + MISC + 1024;
  // TMEM columns: O^T [0, NACC N), S^T [NACC N, (NACC + 2) N), K codes [K_COL + 64 b, +64),
  // V^T codes [V_COL + 64 b, +64) (two f16 per column)
  static constexpr int K_COL = 128;
  static constexpr int V_COL = K_COL + 64 * NBK;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = tk_idesc(128, N, false, false, false);
  static constexpr uint32_t IDESC_PV = tk_idesc(128, N, false, false, true);
  // The two softmax halves take alternate stages, each over all N rows with
  // its own running maxima and O^T accumulator (merged in the epilogue), so
  // a stage's softmax chain overlaps the next one's.
  static constexpr int NH = N;                         // query rows per softmax thread
  static constexpr int NACC = 2;                       // O^T accumulators (one per softmax half)
  // 32-row tiles: the softmax threads hold 32 rows' scores, sums and
  // corrections, more than the 96 registers a thread has at launch, so the
  // softmax warpgroups (warps 0-3, 8-11) take registers from the other three:
  // 2 x 128 x 152 + 3 x 128 x 56 = 60,416 <= 640 x 96 (the launcher checks
  // the 96).
  static constexpr bool kRegSplit = N == 32;
  static constexpr int kSoftRegs = 152, kOtherRegs = 56, kLaunchRegs = 96;
  static_assert(!kRegSplit || 2 * 128 * kSoftRegs + 3 * 128 * kOtherRegs <= 640 * kLaunchRegs, "register pool");
  static_assert((NACC + 2) * N <= K_COL, "tensor-memory budget");
  static_assert(V_COL + 64 * NBV <= TMEM_COLS, "tensor-memory budget");
  static_assert(NS >= 3, "the ring needs a few stages");
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0, "128-byte-swizzled tiles are 1024-aligned");
  static_assert(ST_OFF % 512 == 0 && STAGE % 512 == 0 && K_SLOT % 128 == 0, "64-byte-swizzled records");
  static_assert(REC % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert(BYTES <= 227 * 1024, "shared-memory budget");
};

// Running maximum of a row before its first visible key (log2 domain).
constexpr float kNoMax = -1e30f;

// Byte offset, inside a stage (stages start on 512-byte boundaries), of logical byte `o` of a record
// copied with the 64-byte swizzle: the 16-byte unit index (bits 4-5) is XORed
// with bits 7-8 of the offset.
__device__ __forceinline__ uint32_t sw64(uint32_t o) { return o ^ (((o >> 7) & 3u) << 4); }

template <int N, int PS>
__global__ void __launch_bounds__(640, 1)
    pa_partition_u8(const __grid_constant__ CUtensorMap tmK, const PartArgs a) {
  using C = U8Cfg<N, PS>;
  constexpr int D = C::D;
  constexpr int NH = C::NH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qt = smem + C::Q_OFF;
  uint8_t* pt = smem + C::P_OFF;
  float4* side_buf = reinterpret_cast<float4*>(smem + C::SIDE_OFF);   // [NBV][SK]
  int32_t* blk = reinterpret_cast<int32_t*>(smem + C::BLK_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::MISC_OFF);
  uint64_t* full_k = bars;               // [NS] stage's K records landed
  uint64_t* full_v = full_k + C::NS;     // [NS] stage's V records landed
  uint64_t* empty = full_v + C::NS;      // [NS] stage converted (8 converter warps)
  uint64_t* kfull = empty + C::NS;       // [NBK] K codes in TMEM (8 converter warps)
  uint64_t* kfree = kfull + C::NBK;      // [NBK] K codes consumed (MMA commit after S^T)
  uint64_t* vfull = kfree + C::NBK;      // [NBV] V^T codes in TMEM, side terms written (8 converter warps)
  uint64_t* vfree = vfull + C::NBV;      // [NBV] V^T codes consumed (MMA commit after PV)
  uint64_t* s_full = vfree + C::NBV;     // [2] S^T buffer written (MMA commit)
  uint64_t* s_free = s_full + 2;         // [2] S^T buffer read (8 softmax warps)
  uint64_t* p_full = s_free + 2;         // [2] P'^T buffer written (8 softmax warps)
  uint64_t* pv_done = p_full + 2;        // [2] PV that read that P'^T buffer done (MMA commit)
  float* m_sm = reinterpret_cast<float*>(smem + C::MISC_OFF + 512);   // [2][64] row reference maxima (per half)
  float* xch = m_sm + 128;                                            // [8][64] per-warp row values
  float* m_next = xch + 512;                                          // [2][64]
  float* alpha_sm = m_next + 128;                                     // [2][64]
  long long* rowoff = reinterpret_cast<long long*>(alpha_sm + 128);   // [64]
  float* qsum_sm = reinterpret_cast<float*>(rowoff + 64);             // [64] sum_d of each f16 query row
  float* xch2 = qsum_sm + 64;                                         // [8][64] second exchange
  uint32_t* tree_rows = reinterpret_cast<uint32_t*>(xch2 + 512);      // [8] rows that see new token k
  float* thr_sm = reinterpret_cast<float*>(tree_rows + 8);            // [2][64] maxima + 8: the rescale thresholds
  __shared__ uint32_t s_tmem;
  __shared__ int s_bad, s_timeout;

  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3, hh = warp >> 3;                  // TMEM lane quarter, half
  const bool soft = warp < 16 && (warp & 4) == 0;           // softmax warps 0-3, 8-11
  const bool conv = warp < 16 && (warp & 4) != 0;           // converter warps 4-7, 12-15
  const int st_id = hh * 128 + q4 * 32 + lane;              // index among the 256 threads of a role
  // While the previous kernel may still be running (programmatic dependent
  // launch), warm L2 with the sequence metadata and this partition's
  // block-table slice (prefetches only: every value the kernel uses is
  // loaded after griddepcontrol.wait).
  if (warp == 16 && a.window == 0) {
    if (lane == 0) {
      prefetch_l2(a.begins + b);
      prefetch_l2(a.past_lens + b);
    }
    const long long lpg = (static_cast<long long>(p) * a.part_tokens) >> a.ps_log2;
    const int n = static_cast<int>(min(static_cast<long long>(a.part_tokens >> a.ps_log2),
                                       max(0LL, static_cast<long long>(a.max_blocks) - lpg)));
    for (int j = 32 * lane; j < n; j += 32 * 32) prefetch_l2(a.block_tables + static_cast<size_t>(b) * a.max_blocks + lpg + j);
  }
  // Set-up that reads no input -- barriers, tensor memory, the tensor map's
  // descriptor -- also runs before the wait.
  if (threadIdx.x == 160) {
    s_bad = 0;
    s_timeout = 0;
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full_k[i], 1);
      mbar_init(&full_v[i], 1);
      mbar_init(&empty[i], 8);
    }
    for (int i = 0; i < C::NBK; ++i) {
      mbar_init(&kfull[i], 8);
      mbar_init(&kfree[i], 1);
    }
    for (int i = 0; i < C::NBV; ++i) {
      mbar_init(&vfull[i], 8);
      mbar_init(&vfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);  // the softmax half reading / writing stage s
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 16 && lane == 0) prefetch_tensormap(&tmK);
  tc_fence_before();
  __syncthreads();  // barriers and the TMEM address published
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait_primary();  // inputs and outputs may belong to the previous kernel
  // Without a window a partition's first page is p * part_tokens / page_size
  // whatever the sequence's length, so its block-table slice is fetched
  // before the sequence's bounds are known.
  const bool prefetch = (warp == 16 && a.window == 0);
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
  const int lp0 = kstart / PS;
  const int npages = (kend - 1) / PS - lp0 + 1;
  const int n_stages = (kend - kstart + C::SK - 1) / C::SK;
  const int R = si.T * a.G;
  const float sl2 = a.scale_log2;

  // Stage s's copies from a producer warp, one lane per page: the K records
  // (warp 16, one TMA instruction) or the V records (warp 19, one bulk
  // instruction), each half under its own mbarrier.
  // id_of(j) gives the checked block id of the partition's page j.
  const bool k_producer = warp == 16;
  auto issue_stage = [&](int s, auto id_of) {
    const int slot = s % C::NS;
    const int key0 = kstart + s * C::SK;
    const int npg = (min(C::SK, kend - key0) + PS - 1) / PS;
    uint8_t* st = smem + C::ST_OFF + slot * C::STAGE;
    uint64_t* bar = k_producer ? &full_k[slot] : &full_v[slot];
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(npg * C::REC));
    __syncwarp();
    if (lane < npg) {
      const int lp = key0 / PS + lane;
      const int id = id_of(lp - lp0);
      if (k_producer) {
        tma_load_4d(st + lane * C::K_SLOT, &tmK, 0, 0, g, id, bar);
        if (a.trace != nullptr)
          atomicAdd(a.trace + (static_cast<size_t>(b) * a.Hkv + g) * a.max_blocks + lp, id + 1);
      } else {
        bulk_load(st + C::K_AREA + lane * C::REC,
                  a.v_bytes + (static_cast<size_t>(id) * a.Hkv + g) * static_cast<size_t>(C::REC), C::REC, bar);
      }
    }
    __syncwarp();
  };

  // ---- set-up: the first stages' copies go out as soon as their block ids
  // are known; meanwhile tensor memory is allocated and Q staged.  A bad id
  // is reported, clamped to page 0 (every copy stays in bounds) and the
  // partition's result discarded. ----
  const int32_t* bt_row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + lp0;
  if (warp == 16) {
    int bad = 0;
    if (prefetch) {
      cp_async_wait_all();
      __syncwarp();
    }
    auto checked = [&](int j) {
      int id = prefetch ? blk[j] : ld_once(bt_row + j);
      if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
        bad = 1;
        id = 0;
      }
      return id;
    };
    for (int s = 0; s < min(C::NS, n_stages); ++s) issue_stage(s, checked);
    // the later stages' ids, checked once, for both producers
    for (int j = C::NS * C::PPS + lane; j < npages; j += 32) blk[j] = checked(j);
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      s_bad = 1;
      atomicOr(a.status, PA_STATUS_BLOCK_ID);
    }
    __syncwarp();
    bar_sync_n(2, 64);  // checked ids published to the V producer
  } else if (warp == 19) {
    // the V producer's first stages read the ids itself (the K producer
    // reports bad ones)
    auto clamped = [&](int j) {
      const int id = ld_once(bt_row + j);
      return static_cast<unsigned>(id) < static_cast<unsigned>(a.num_blocks) ? id : 0;
    };
    for (int s = 0; s < min(C::NS, n_stages); ++s) issue_stage(s, clamped);
    bar_sync_n(2, 64);
  }
  if (soft) {
    // Q rows -> f16, K-major swizzled tile (rows R..N-1 zero); then the sum of
    // each f16 row, in head-dim order
    for (int idx = st_id; idx < N * (D / 8); idx += 256) {
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
          const __half2 hh2 = __floats2half2_rn(f.x, f.y);
          h[e] = *reinterpret_cast<const uint32_t*>(&hh2);
        }
        v = make_uint4(h[0], h[1], h[2], h[3]);
      }
      *reinterpret_cast<uint4*>(qt + ((u16 >> 3) * N + n) * 128 + swz(u16 & 7, n)) = v;
    }
    // No key seen yet: a finite floor far below any score (a row's first
    // visible key always exceeds it by more than the rescale threshold; the
    // weights 2^(x - m) of masked keys (x = -inf) stay 0 and the rescale
    // factor 2^(floor - m) of the first rescale is 0).
    if (st_id < 128) {
      m_sm[st_id] = kNoMax;
      thr_sm[st_id] = kNoMax + 8.f;
    }
    fence_proxy_async();  // the Q tile is read by the tensor cores
    bar_sync_n(1, 256);
    if (st_id < N) {
      const int n = st_id;
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
    if (st_id >= 64 && st_id < 64 + PA_MAX_QUERY_LEN) {
      // tree masks: the rows that see new token k (row n = token n / G)
      const int k = st_id - 64;
      uint32_t rows = 0;
      if (a.tree_mask != nullptr)
        for (int n = 0; n < R; ++n) rows |= ((ld_once_u8(a.tree_mask + si.t0 + n / a.G) >> k) & 1u) << n;
      tree_rows[k] = rows;
    }
  }
  // Q tile and row sums published to all warps
  __syncthreads();
  const uint32_t tm_o = tmem;            // O^T accumulators: lane = head dim, column = row
  const uint32_t tm_s0 = tmem + C::NACC * N;  // S^T buffers: lane = key, column = row
  const uint32_t tm_k = tmem + C::K_COL; // K codes + 1024: lane = key, two f16 per column
  const uint32_t tm_v = tmem + C::V_COL; // V^T codes: lane = head dim, two keys per column
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  bool ok = true;

  // The roles part here; each ends at the kernel's two closing barriers, so
  // that a warpgroup's register budget holds from its role to its exit.
  if (!soft) {
  if constexpr (C::kRegSplit) regs_decrease<C::kOtherRegs>();
  if (conv) {
    // =========================== converters =================================
    const int ct = q4 * 32 + lane;                             // key (K) and head dim (V^T), 0..127
    const int pi = ct / PS, kk = ct % PS;
    const uint32_t k_row = static_cast<uint32_t>(pi * C::K_SLOT + kk * 128 + 64 * hh);  // this half of the row
    const uint32_t sc = hh == 0 ? static_cast<uint32_t>(pi * C::K_SLOT + 128 * PS + 2 * kk)
                                : static_cast<uint32_t>(C::K_AREA + pi * C::REC + 128 * PS + 2 * kk);
    const __half2 k1024 = __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    // key ct's dequantisation terms (K for h = 0, V for h = 1); zero
    // outside every row's range and past the partition (there the scales
    // may be garbage, even NaN)
    auto side_terms = [&](const uint8_t* st, int s, int vb) {
      const int key = kstart + s * C::SK + ct;
      const bool in = key >= si.klo && key <= si.khi && key < kend;
      const float sv = __half2float(*reinterpret_cast<const __half*>(st + (hh == 0 ? sw64(sc) : sc)));
      const float zv = __half2float(*reinterpret_cast<const __half*>(st + (hh == 0 ? sw64(sc + 2 * PS) : sc + 2 * PS)));
      float2 t = hh == 0 ? make_float2(sv * sl2, zv + 1024.f) : make_float2(sv, zv);
      if (!in) t = make_float2(0.f, 0.f);
      reinterpret_cast<float2*>(side_buf + vb * C::SK + ct)[hh] = t;
    };
    for (int s = 0; s < n_stages && ok; ++s) {
      const int kb = s % C::NBK, vb = s % C::NBV, slot = s % C::NS;
      if (!mbar_wait(&full_k[slot], (s / C::NS) & 1) ||
          (s >= C::NBK && !mbar_wait(&kfree[kb], ((s / C::NBK) - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint8_t* st = smem + C::ST_OFF + slot * C::STAGE;
      {
        // head dims [64h, 64h + 64) of key ct's K codes -> (1024 + code) as
        // f16 pairs; column j of the half holds dims 64h + 2j, 64h + 2j + 1
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 x = *reinterpret_cast<const uint4*>(st + sw64(k_row + 16 * u));
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            w[8 * u + 2 * e] = __byte_perm(xs[e], 0x64646464u, 0x4140u);
            w[8 * u + 2 * e + 1] = __byte_perm(xs[e], 0x64646464u, 0x4342u);
          }
        }
        tmem_st32_nowait(tm_k + kb * 64 + 32 * hh + lane_off, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kfull[kb]);  // S^T(s) may start
      if (!mbar_wait(&full_v[slot], (s / C::NS) & 1) ||
          (s >= C::NBV && !mbar_wait(&vfree[vb], ((s / C::NBV) - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the side terms' slot was last read by the softmax of stage s - NBV,
      // which finished before PV(s - NBV) was issued
      side_terms(st, s, vb);
      {
        // V^T: head dim ct of keys [64h, 64h + 64) -> exact f16 codes, keys
        // 64h + 2j, 64h + 2j + 1 in column j of the half.  V records hold
        // their codes dim-major, so the 16 codes of one head dim over 16 keys
        // of a page are one 16-byte load.
        uint32_t w[32];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int k0 = 64 * hh + 16 * m;
          const uint4 x = *reinterpret_cast<const uint4*>(st + C::K_AREA + (k0 / PS) * C::REC + ct * PS + (k0 % PS));
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t h0 = __byte_perm(xs[e], 0x64646464u, 0x4140u);
            uint32_t h1 = __byte_perm(xs[e], 0x64646464u, 0x4342u);
            const __half2 c0 = __hsub2(*reinterpret_cast<const __half2*>(&h0), k1024);
            const __half2 c1 = __hsub2(*reinterpret_cast<const __half2*>(&h1), k1024);
            w[8 * m + 2 * e] = *reinterpret_cast<const uint32_t*>(&c0);
            w[8 * m + 2 * e + 1] = *reinterpret_cast<const uint32_t*>(&c1);
          }
        }
        tmem_st32_nowait(tm_v + vb * 64 + 32 * hh + lane_off, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vfull[vb]);
        mbar_arrive(&empty[slot]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      atomicOr(a.status, PA_STATUS_TIMEOUT);
      atomicOr(&s_timeout, 1);
    }
  } else if (warp == 16 || warp == 19) {
    // =========================== producers ==================================
    int issued = min(C::NS, n_stages);
    for (int s = C::NS; s < n_stages && ok; ++s) {
      // the slot is free once the eight converter warps are done with stage s - NS
      if (!mbar_wait(&empty[s % C::NS], ((s / C::NS) - 1) & 1)) {
        ok = false;
        break;
      }
      issue_stage(s, [&](int j) { return blk[j]; });
      issued = s + 1;
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
      // let this warp's copies in flight land before the CTA can retire
      uint64_t* mine = k_producer ? full_k : full_v;
      for (int s = max(0, issued - C::NS); s < issued; ++s) mbar_wait(&mine[s % C::NS], (s / C::NS) & 1);
    }
  } else if (warp == 17) {
    // =========================== S^T MMA issuer =============================
    if (lane == 0) {
      const uint32_t q_base = smem_u32(qt);
      bool fine = true;
      for (int ns = 0; ns < n_stages && fine; ++ns) {
        const int kb = ns % C::NBK, sb = ns & 1;
        fine = mbar_wait(&kfull[kb], (ns / C::NBK) & 1);
        if (fine && ns >= 2) fine = mbar_wait(&s_free[sb], ((ns >> 1) - 1) & 1);
        if (!fine) break;
        tc_fence_after();
#pragma unroll
        for (int kc = 0; kc < D / 16; ++kc) {
          const uint64_t bd = sw128_desc(q_base + (kc >> 2) * N * 128 + 32 * (kc & 3), 16, 1024);
          tc_mma_ta(tm_s0 + sb * N, tm_k + kb * 64 + 8 * kc, bd, C::IDESC_S, kc > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        tc_commit(&kfree[kb]);
      }
      if (!fine) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  } else if (warp == 18) {
    // =========================== PV MMA issuer ==============================
    if (lane == 0) {
      bool fine = true;
      for (int np = 0; np < n_stages && fine; ++np) {
        const int pb = np & 1, vb = np % C::NBV;
        fine = mbar_wait(&p_full[pb], (np >> 1) & 1);
        if (!fine) break;
        tc_fence_after();
        const uint32_t p_base = smem_u32(pt + pb * C::P_BYTES);
#pragma unroll
        for (int j = 0; j < C::SK / 16; ++j) {
          const uint64_t bd = sw128_desc(p_base + j * 16 * 128, 0, 1024);
          tc_mma_ta(tm_o + (np & 1) * N, tm_v + vb * 64 + 8 * j, bd, C::IDESC_PV,
                    (np >= C::NACC || j > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[pb]);
        tc_commit(&vfree[vb]);
      }
      if (!fine) {
        atomicOr(a.status, PA_STATUS_TIMEOUT);
        atomicOr(&s_timeout, 1);
      }
    }
    __syncwarp();
  }
  __syncthreads();  // every role is done
  __syncthreads();  // the softmax warps' epilogue is done
  return;
  }

  // =========================== softmax warps (keys) ==========================
  if constexpr (C::kRegSplit) regs_increase<C::kSoftRegs>();
  float l[NH], zc[NH];
  {
    const int kq = q4 * 32 + lane;     // key of the stage
    const int n0 = 0;                  // this thread's rows [n0, n0 + NH): all of them
    const int hbar = 3 + hh;           // named barrier of this half's four warps
    // this half's running state: its own maxima and accumulator
    float* ms = m_sm + hh * 64;
    float* mnx = m_next + hh * 64;
    float* al = alpha_sm + hh * 64;
    float* th = thr_sm + hh * 64;
    const uint32_t tm_og = tm_o + hh * N;
    constexpr int kStep = 2;           // stages between this half's stages
#pragma unroll
    for (int e = 0; e < NH; ++e) {
      l[e] = 0.f;
      zc[e] = 0.f;
    }
    const bool tree = a.tree_mask != nullptr;
    for (int s = hh; s < n_stages; s += kStep) {
      const int sb = s & 1, vb = s % C::NBV;
      if (ok) ok = mbar_wait(&s_full[sb], (s >> 1) & 1);
      tc_fence_after();
      float v[NH];
      tmem_ld_small<NH>(tm_s0 + sb * N + n0 + lane_off, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      // this key's dequantisation terms (written by the converters before vfull)
      if (ok) ok = mbar_wait(&vfull[vb], (s / C::NBV) & 1);
      const float4 sd = side_buf[vb * C::SK + kq];

      // Every row sees every key of the stage (the common case: past keys
      // inside every row's window and the partition) -- the same for all
      // threads, so the per-key row mask is skipped.
      const int k0 = kstart + s * C::SK;
      const bool stage_clean = !tree && k0 + C::SK - 1 <= si.L && k0 + C::SK <= kend &&
                               (a.window == 0 || k0 - si.L + a.window >= si.T);
      uint32_t vrows = 0xffffffffu;
      if (!stage_clean) {
        const int key = k0 + kq;
        const int dk = key - si.L;
        // rows that see this key, as a bit set: [nlo, nhi) (the causal limit
        // and the window), or for a tree mask the window and the rows whose
        // mask names this new token
        const int nlo = (dk > 0 && !tree) ? dk * a.G : 0;
        int nhi = R;
        if (a.window > 0) nhi = min(R, max(0, (dk + a.window) * a.G));
        if (key >= kend) nhi = 0;  // past the partition: the next partition's keys
        const uint32_t below_hi = nhi >= 32 ? 0xffffffffu : ((1u << nhi) - 1u);
        const uint32_t below_lo = nlo >= 32 ? 0xffffffffu : ((1u << nlo) - 1u);
        vrows = below_hi & ~below_lo;
        if (tree && dk >= 0) vrows &= (dk < PA_MAX_QUERY_LEN) ? tree_rows[dk] : 0u;
      }
      bool need = false;
#pragma unroll
      for (int e4 = 0; e4 < NH; e4 += 4) {
        const float4 t4 = *reinterpret_cast<const float4*>(th + n0 + e4);
        const float4 qq = *reinterpret_cast<const float4*>(qsum_sm + n0 + e4);
        const float tt[4] = {t4.x, t4.y, t4.z, t4.w};
        const float qs[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = fmaf(-sd.y, qs[e], v[e4 + e]) * sd.x;
          if (!stage_clean) x = ((vrows >> (n0 + e4 + e)) & 1u) ? x : -INFINITY;
          v[e4 + e] = x;
          need |= x > tt[e];
        }
      }
      // A half's four warps share one set of running maxima (all rows of
      // the half's stages), so the rescale decision and the new maxima
      // involve only them (named barrier 3 + h).
      if (bar_any(hbar, 128, need)) {
        const int xw = hh * 4 + q4;  // this warp's slot in the exchange
        float t[NH];
#pragma unroll
        for (int e = 0; e < NH; ++e) t[e] = v[e];
        const float tm = warp_reduce_split<NH>(t, lane, OpMax());  // row lane / (32 / NH)
        if (lane % (32 / NH) == 0) xch[xw * 64 + n0 + lane / (32 / NH)] = tm;
        bar_sync_n(hbar, 128);
        const int hr = q4 * 32 + lane;  // a row of this half, for the first NH threads
        if (hr < NH) {
          const int n = n0 + hr;
          const float rm = fmaxf(fmaxf(xch[(hh * 4) * 64 + n], xch[(hh * 4 + 1) * 64 + n]),
                                 fmaxf(xch[(hh * 4 + 2) * 64 + n], xch[(hh * 4 + 3) * 64 + n]));
          const float mo = ms[n];
          const float mn = rm > mo + 8.f ? rm : mo;
          mnx[n] = mn;
          al[n] = (mn == mo) ? 1.f : ex2(mo - mn);
        }
        bar_sync_n(hbar, 128);
#pragma unroll
        for (int e = 0; e < NH; ++e) {
          l[e] *= al[n0 + e];
          zc[e] *= al[n0 + e];
        }
        if (hr < NH) {
          ms[n0 + hr] = mnx[n0 + hr];
          th[n0 + hr] = mnx[n0 + hr] + 8.f;
        }
        if (s >= kStep) {
          // rescale this half's columns of its O^T accumulator once the
          // previous PV into it has landed
          const int sp = s - kStep;
          if (ok) ok = mbar_wait(&pv_done[sp & 1], (sp >> 1) & 1);
          tc_fence_after();
          float o[NH];
          tmem_ld_small<NH>(tm_og + n0 + lane_off, o);
#pragma unroll
          for (int e = 0; e < NH; ++e) o[e] *= al[n0 + e];
          tmem_st_small<NH>(tm_og + n0 + lane_off, reinterpret_cast<const uint32_t*>(o));
          tc_fence_before();
        }
        bar_sync_n(hbar, 128);
      }
      // weights times the key's V scale, rounded to f16 as the MMA reads them
      // (8 rows = one 16-byte unit of this key's P'^T row at a time); the
      // zero-point correction uses the rounded values.  The P'^T buffer is
      // free once the PV two stages back has finished.
      if (s >= 2 && ok) ok = mbar_wait(&pv_done[sb], ((s >> 1) - 1) & 1);
      uint8_t* prow = pt + sb * C::P_BYTES + kq * 128;
      const uint16_t vz_bits = __half_as_ushort(__float2half_rn(sd.w));  // the stored f16 zero-point
#pragma unroll
      for (int u = 0; u < NH / 8; ++u) {
        const float4 ma = *reinterpret_cast<const float4*>(ms + n0 + 8 * u);
        const float4 mb = *reinterpret_cast<const float4*>(ms + n0 + 8 * u + 4);
        const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int i = 8 * u + e;
          const float p0 = ex2(v[i] - mm[e]), p1 = ex2(v[i + 1] - mm[e + 1]);
          l[i] += p0;
          l[i + 1] += p1;
          const __half2 h = __floats2half2_rn(p0 * sd.z, p1 * sd.z);
          zc[i] = fma_f16_f32(__half_as_ushort(__low2half(h)), vz_bits, zc[i]);
          zc[i + 1] = fma_f16_f32(__half_as_ushort(__high2half(h)), vz_bits, zc[i + 1]);
          pk[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(prow + swz(n0 / 8 + u, kq)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
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
  {
    // ---- epilogue, alternating halves: each half's row sums and corrections
    // over its stages' keys, the two halves merged (log-sum-exp), then O^T ----
    const int xw = hh * 4 + q4;
    const int dd = q4 * 32 + lane;  // head dim of this thread's O^T lane
    {
      const float t = warp_reduce_split<NH>(l, lane, OpAdd());  // row lane / (32 / NH)
      const float z = warp_reduce_split<NH>(zc, lane, OpAdd());
      if (lane % (32 / NH) == 0) {
        xch[xw * 64 + lane / (32 / NH)] = t;
        xch2[xw * 64 + lane / (32 / NH)] = z;
      }
    }
    bar_sync_n(1, 256);
    const bool poisoned = s_bad != 0 || s_timeout != 0;
    float* linv = alpha_sm;        // [64]
    float* zrow = m_next;          // [64]
    float* wa = alpha_sm + 64;     // half 0's weight per row
    float* wb = m_next + 64;       // half 1's weight per row
    if (st_id < R) {
      const int n = st_id;
      const float la = (xch[0 * 64 + n] + xch[1 * 64 + n]) + (xch[2 * 64 + n] + xch[3 * 64 + n]);
      const float lb = (xch[4 * 64 + n] + xch[5 * 64 + n]) + (xch[6 * 64 + n] + xch[7 * 64 + n]);
      const float za = (xch2[0 * 64 + n] + xch2[1 * 64 + n]) + (xch2[2 * 64 + n] + xch2[3 * 64 + n]);
      const float zb = (xch2[4 * 64 + n] + xch2[5 * 64 + n]) + (xch2[6 * 64 + n] + xch2[7 * 64 + n]);
      const float ma = m_sm[n], mb = m_sm[64 + n];
      const float M = fmaxf(ma, mb);
      const float wA = ex2(ma - M), wB = ex2(mb - M);
      const float lt = wA * la + wB * lb;
      zrow[n] = wA * za + wB * zb;
      wa[n] = wA;
      wb[n] = wB;
      const long long row = static_cast<long long>(si.t0 + n / a.G) * a.Hq + g * a.G + n % a.G;
      if (si.nparts == 1) {
        rowoff[n] = row * D;
        linv[n] = (poisoned || !(lt > 0.f)) ? 0.f : 1.f / lt;
      } else {
        rowoff[n] = (prow(row, si, a.Hq) * a.num_parts + p) * D;
        a.pm[prow(row, si, a.Hq) * a.num_parts + p] = M;
        a.pl[prow(row, si, a.Hq) * a.num_parts + p] = poisoned ? -1.f : lt;
      }
    }
    bar_sync_n(1, 256);
    tc_fence_after();
    // this thread: head dim dd of rows [hN/2, (h+1)N/2), both accumulators
    // (the second one holds nothing when the partition has a single stage)
    constexpr int RH = N / 2;
    const int r0 = hh * RH;
    const bool has_b = n_stages >= 2;
    float oa[RH], ob[RH];
    tmem_ld_small<RH>(tm_o + r0 + lane_off, oa);
    tmem_ld_small<RH>(tm_o + N + r0 + lane_off, ob);
#pragma unroll
    for (int e = 0; e < RH; ++e) {
      const int n = r0 + e;
      if (n < R) {
        const float o = fmaf(wa[n], oa[e], has_b ? wb[n] * ob[e] : 0.f) - zrow[n];
        if (si.nparts > 1) a.po[rowoff[n] + dd] = o;
        else store_out(a.out, a.out_dtype, rowoff[n] + dd, poisoned ? 0.f : o * linv[n]);
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
