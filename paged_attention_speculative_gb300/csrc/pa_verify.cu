// pa_verify.cu — C-ABI implementation: argument checks, the partition-count
// heuristic, TMA descriptor set-up and the kernel launches.
//
// The heuristic follows the split-KV idea of the pages (OpenVINO issue 38153,
// "Cause": 256-token partitions of the single-token stage; dual-radeon-vllm
// article: the 3D kernel splits a long KV sequence into segments reduced in
// parallel, and a fix derives its threshold from the SM count): the key range
// every (sequence, KV head) must stream is cut into equal partitions so that
// the grid fills the GPU's SMs about once, partitions never shrink below the
// size at which per-token partials would cost more than ~10 % of the KV bytes,
// and the split does not depend on how many query tokens a sequence brings.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/pa_verify.h"
#include "pa_combine.cuh"
#include "pa_launch.h"
#include "pa_partition_f32.cuh"

namespace {

using pa::CombineArgs;
using pa::PartArgs;

constexpr size_t kStatusBytes = 256;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
long long round_up(long long a, long long q) { return ceil_div(a, q) * q; }

int dtype_bytes(pa_dtype t) { return t == PA_F32 ? 4 : (t == PA_U8 ? 1 : 2); }

// Optional override of the partition kernel, read once: "tc" forces the
// 16-bit rows-on-M tensor-memory kernel wherever it applies, "mma" the
// warp-level one (16-bit and u8 caches); unset = chosen by shape.
int env_kernel_choice() {
  static const int v = [] {
    const char* s = std::getenv("PA_VERIFY_KERNEL");
    if (s == nullptr) return 0;
    if (std::strcmp(s, "tc") == 0) return 2;
    if (std::strcmp(s, "mma") == 0) return 1;
    return 0;
  }();
  return v;
}

// Optional tuning override of the partition size (keys), read once.
int env_part_tokens() {
  static const int v = [] {
    const char* s = std::getenv("PA_VERIFY_PART_TOKENS");
    return s ? std::atoi(s) : 0;
  }();
  return v;
}

// Optional tuning override of the warp-level kernel's n-tiles per warp (1 or 2), read once.
int env_row_tiles() {
  static const int v = [] {
    const char* s = std::getenv("PA_VERIFY_ROW_TILES");
    const int n = s ? std::atoi(s) : 0;
    return (n == 1 || n == 2) ? n : 0;
  }();
  return v;
}

// Optional tuning override of the prefill blocks' key pieces (1..32), read once.
int env_prefill_splits() {
  static const int v = [] {
    const char* s = std::getenv("PA_PREFILL_SPLITS");
    const int n = s ? std::atoi(s) : 0;
    return (n >= 1 && n <= 32) ? n : 0;
  }();
  return v;
}

// Optional tuning override of the prefill kernel's rows per CTA (128 or 256), read once.
int env_prefill_rows() {
  static const int v = [] {
    const char* s = std::getenv("PA_PREFILL_ROWS");
    const int n = s ? std::atoi(s) : 0;
    return (n == 128 || n == 256) ? n : 0;
  }();
  return v;
}

int mma_kind(pa_dtype kv) { return kv == PA_BF16 ? pa::KV_BF16 : (kv == PA_F16 ? pa::KV_F16 : pa::KV_U8); }

pa::MmaKernelInfo mma_info(int D, int kind, int nt, bool* ok) {
  if (D == 64) return pa::mma_info_d64(kind, nt, ok);
  if (D == 128) return pa::mma_info_d128(kind, nt, ok);
  if (D == 256) return pa::mma_info_d256(kind, nt, ok);
  *ok = false;
  return pa::MmaKernelInfo{0, 0, 0};
}

// Argument checks shared by every entry point; fills the plan.
int make_plan(const pa_dims* d, int32_t max_ctx, int32_t window, pa_dtype kv, int32_t num_sms, pa_plan* plan) {
  if (d == nullptr || plan == nullptr) return PA_ERR_NULL;
  std::memset(plan, 0, sizeof(*plan));
  if (d->num_seqs < 1 || d->num_seqs > 65535 || d->total_tokens < 0 || d->num_q_heads < 1 ||
      d->num_kv_heads < 1 || d->num_kv_heads > 65535 || d->num_q_heads % d->num_kv_heads != 0 ||
      d->num_blocks < 1 || d->max_blocks_per_seq < 1 || window < 0 || num_sms < 1)
    return PA_ERR_SHAPE;
  const int D = d->head_dim;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_HEAD_DIM;
  if (kv == PA_U8 && D == 64) return PA_ERR_HEAD_DIM;
  const int ps = d->page_size;
  if (!pow2(ps) || ps > 256) return PA_ERR_PAGE_SIZE;
  // Pages of 1, 2 or 4 tokens: fp32 caches (the FFMA kernel looks every key
  // up anyway), 16-bit caches with head_dim <= 128 (the tensor-memory
  // kernel's cp.async-gather producer) and with head_dim 256 (the warp-level
  // kernel's per-key bulk copies).  The other kernels stage whole pages with
  // TMA boxes and take 8 tokens or more.
  const bool small_pages = ps < pa::kGatherBelowPageSize;
  if (small_pages && !(kv == PA_F32 || kv == PA_BF16 || kv == PA_F16)) return PA_ERR_PAGE_SIZE;
  // u8 V pages are copied as [head dim][key] boxes at least 16 keys wide
  if (kv == PA_U8 && ps < 16) return PA_ERR_PAGE_SIZE;
  const pa_dtype qd = d->q_dtype, od = d->out_dtype;
  if (od != PA_F32 && od != PA_F16 && od != PA_BF16) return PA_ERR_DTYPE;
  bool combo = (kv == PA_F32 && (qd == PA_F32 || qd == PA_F16 || qd == PA_BF16)) ||
               (kv == PA_BF16 && qd == PA_BF16) || (kv == PA_F16 && qd == PA_F16) ||
               (kv == PA_U8 && (qd == PA_BF16 || qd == PA_F16));
  if (!combo) return PA_ERR_DTYPE;
  if (d->total_tokens > 0 &&
      (max_ctx < 1 || static_cast<long long>(max_ctx) > static_cast<long long>(d->max_blocks_per_seq) * ps))
    return PA_ERR_CONTEXT;
  if (max_ctx < 0) return PA_ERR_CONTEXT;

  const int G = d->num_q_heads / d->num_kv_heads;
  const int tmax = std::min(PA_MAX_QUERY_LEN, std::max(d->total_tokens, 1));
  const long long rows = static_cast<long long>(G) * tmax;
  int kernel = (kv == PA_F32) ? 1 : 0;
  int nt = 0, sk = 64, smem = 0, ctas_per_sm = 4;
  // 16-bit caches go to the tensor-memory path: its cost per key does not
  // grow with the row count (measured: T=4 x 4 heads and T=8 x 8 heads cost
  // 1.01-1.05x a single-token step), and with head_dim 128 it is also the
  // faster one for a single token (T=1 x 4 heads at 32k keys: 28.3 us vs
  // 29.4 us on the warp-level kernel).  With head_dim 64 the warp-level
  // kernel stays ahead below 8 rows (10.8 vs 10.9 us).
  const bool tc16 = (kv == PA_BF16 || kv == PA_F16) && (D == 64 || D == 128);
  // Small pages always take the rows-on-M tensor-memory kernel (16-bit
  // caches, head_dim <= 128) or the warp-level one (head_dim 256).
  const int choice = small_pages ? (D == 256 ? 1 : 2) : env_kernel_choice();
  // u8 caches with head_dim 128, pages of 16 / 32 / 64 tokens and up to 32
  // query rows per KV head take the u8 tensor-memory kernel: each code is
  // converted once per stage whatever the row count, so its cost does not
  // grow with the query tokens.  Other u8 shapes take the warp-level kernel.
  if (kv == PA_U8 && D == 128 && rows <= 32 && (ps == 16 || ps == 32 || ps == 64) && choice != 1) {
    const int n = rows <= 16 ? 16 : 32;
    bool ok = false;
    pa::MmaKernelInfo info = pa::u8_info(n, ps, &ok);
    if (ok) {
      kernel = 4;
      nt = n;
      sk = info.stage_keys;
      smem = info.smem_bytes;
      ctas_per_sm = info.ctas_per_sm;
    }
  }
  if (kernel == 0 && tc16 && rows <= 64 && choice != 1 && (rows >= 8 || D == 128 || choice == 2)) {
    bool ok = false;
    pa::MmaKernelInfo info = pa::tc_info(D, mma_kind(kv), &ok);
    if (ok) {
      kernel = 2;
      sk = info.stage_keys;
      smem = info.smem_bytes;
      ctas_per_sm = info.ctas_per_sm;
    }
  }
  // more than 64 rows per KV head (head_dim <= 128)
  if (small_pages && kernel != 1 && kernel != 2 && D != 256) return PA_ERR_PAGE_SIZE;
  if (kernel == 0) {
    // one 8-row n-tile per warp keeps a warp's accumulators within the
    // register budget of two CTAs per SM; rows beyond 8 go to more warps
    nt = (D == 256 || rows <= 32) ? 1 : 2;
    if (env_row_tiles() > 0 && D != 256) nt = env_row_tiles();
    const int cap = pa::kConsumerWarps * 8 * nt;
    if (rows > cap) return PA_ERR_UNSUPPORTED;
    bool ok = false;
    pa::MmaKernelInfo info =
        small_pages ? pa::mma_info_d256_gather(mma_kind(kv), &ok) : mma_info(D, mma_kind(kv), nt, &ok);
    if (!ok) return PA_ERR_UNSUPPORTED;
    sk = info.stage_keys;
    smem = info.smem_bytes;
    ctas_per_sm = info.ctas_per_sm;
  }
  // Partitions are whole stages, except on the u8 tensor-memory kernel: its
  // stages may end at a partition boundary (codes are finite and the scales
  // of keys past the boundary are zeroed), so a page quantum evens out the
  // bytes per CTA (32k keys on 152 CTAs: 1728 keys each, not 1792 and a
  // short last partition).
  const long long quantum = kernel == 4 ? ps : std::max(sk, ps);
  const long long ctx = std::max<long long>(max_ctx, 1);
  long long span = window > 0 ? std::min<long long>(ctx, static_cast<long long>(window) + tmax - 1 + ps - 1) : ctx;
  const long long units = static_cast<long long>(d->num_seqs) * d->num_kv_heads;
  const long long per_key = 2LL * D * dtype_bytes(kv) + (kv == PA_U8 ? 8 : 0);
  const long long target = static_cast<long long>(num_sms) * ctas_per_sm;
  long long part = ceil_div(span * units, target);
  const long long min_part = ceil_div(10LL * rows * (D + 2) * 4, per_key);
  part = std::max(part, std::max<long long>(min_part, 2LL * sk));
  if (env_part_tokens() > 0) part = env_part_tokens();
  part = round_up(std::max<long long>(part, 1), quantum);
  part = std::min(part, round_up(span, quantum));
  // kernels that stage the partition's block ids in shared memory take at
  // most kMaxPagesPerCta pages per CTA; the small-page paths look ids up per
  // stage and have no such cap
  const long long page_cap = small_pages ? round_up(span, quantum)
                                         : (static_cast<long long>(pa::kMaxPagesPerCta - 1) * ps / quantum) * quantum;
  part = std::min(part, std::max(page_cap, quantum));
  if (env_part_tokens() <= 0) {
    // Rounding can leave a last wave of CTAs that is mostly empty; a larger
    // partition that needs fewer waves is then cheaper.  Cost = waves x keys
    // per CTA, the serial work of the busiest CTA slot.
    const long long cap = std::min(round_up(span, quantum), std::max(page_cap, quantum));
    auto cost = [&](long long pt) { return ceil_div(ceil_div(span, pt) * units, target) * pt; };
    long long best = part, best_cost = cost(part);
    for (long long cand = part + quantum; cand <= cap && ceil_div(ceil_div(span, best) * units, target) > 1;
         cand += quantum) {
      const long long c = cost(cand);
      if (c < best_cost) {
        best = cand;
        best_cost = c;
      }
    }
    part = best;
  }
  const long long P = ceil_div(span, part);
  if (P > 65535 || P * units > (1LL << 31)) return PA_ERR_UNSUPPORTED;

  plan->num_partitions = static_cast<int32_t>(P);
  plan->part_tokens = static_cast<int32_t>(part);
  plan->stage_keys = sk;
  plan->row_tiles = nt;
  plan->kernel = kernel;
  plan->num_sms = num_sms;
  plan->ctas = static_cast<int32_t>(P * units);
  plan->smem_bytes = smem;
  return PA_OK;
}

// Token slots of the split-KV partials: one per token, or 8 per sequence in
// a mixed call (its verify steps index partials by b * 8 + i).
size_t partial_slots(const pa_dims* d, bool mixed) {
  return mixed ? static_cast<size_t>(d->num_seqs) * PA_MAX_QUERY_LEN : static_cast<size_t>(d->total_tokens);
}

size_t workspace_bytes_for(const pa_dims* d, const pa_plan& plan, bool mixed = false) {
  const size_t rows = partial_slots(d, mixed) * d->num_q_heads * plan.num_partitions;
  return kStatusBytes + align256(rows * d->head_dim * 4) + 2 * align256(rows * 4);
}

struct Workspace {
  uint32_t* status;
  float* po;
  float* pm;
  float* pl;
};

Workspace carve(void* ws, const pa_dims* d, const pa_plan& plan, bool mixed = false) {
  const size_t rows = partial_slots(d, mixed) * d->num_q_heads * plan.num_partitions;
  uint8_t* base = static_cast<uint8_t*>(ws);
  Workspace w;
  w.status = reinterpret_cast<uint32_t*>(base);
  w.po = reinterpret_cast<float*>(base + kStatusBytes);
  w.pm = reinterpret_cast<float*>(base + kStatusBytes + align256(rows * d->head_dim * 4));
  w.pl = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(w.pm) + align256(rows * 4));
  return w;
}

// Row blocks of a mixed call's prefill chunks and the pieces their keys are
// split into, from what the host knows (dims, max_context_len, the window and
// the SM count; the chunks' lengths are device data, so `tiles` is an upper
// bound: every token in full blocks plus one partial block per possible
// chunk).  Blocks are 128 rows (one tile; measured faster than 256-row
// blocks of two ping-ponging tiles at every chunk size since the one-tile
// blocks split their producers and issuers: 2.5k-4k-token chunks 10-24 %,
// same box).  PA_PREFILL_ROWS=256 keeps the two-tile blocks reachable for
// tuning.  When the blocks fill at most half the SMs and every
// piece keeps >= 4096 keys, each block's keys are split into pieces, as many
// as still fit in one wave (measured, chunk alone: 64 tokens at 32k keys
// 361 -> 76 us, 128 tokens at 64k keys 696 -> 247 us).  Blocks that fill a
// wave or more are not split: a split over several waves can add one (512
// tokens at 32k keys in 6 pieces: 376 -> 400 us).  The host bounds the
// pieces (`splits`, the grid's z extent and the partial rows' stride) by the
// fewest blocks the batch can have -- its tokens beyond 8 per sequence -- and
// the kernels count the blocks the batch really has and use as many of the
// pieces as fit in one wave (prefill_pieces); the others exit at once.
struct PrefillGeometry {
  int rows_per_block;
  long long tiles;
  int splits;
};

PrefillGeometry prefill_geometry(const pa_dims* d, int32_t max_ctx, int32_t window, int sms) {
  PrefillGeometry pg;
  const int G = d->num_q_heads / d->num_kv_heads;
  pg.rows_per_block = env_prefill_rows() > 0 ? env_prefill_rows() : 128;
  const long long TQ = pg.rows_per_block / G;
  pg.tiles = ceil_div(d->total_tokens, TQ) +
             std::min<long long>(d->num_seqs, d->total_tokens / (PA_MAX_QUERY_LEN + 1));
  const long long keys = window > 0 ? std::min<long long>(max_ctx, static_cast<long long>(window) + TQ) : max_ctx;
  const long long min_blocks =
      std::max<long long>(1, ceil_div(std::max<long long>(0, d->total_tokens - 8LL * d->num_seqs), TQ));
  const long long S_fit = std::min<long long>(std::min<long long>(16, keys / pa::kPrefillMinPieceKeys),
                                              sms / (min_blocks * d->num_kv_heads));
  int S = static_cast<int>(std::max<long long>(1, S_fit));
  if (env_prefill_splits() > 0) S = env_prefill_splits();
  pg.splits = S;
  return pg;
}

// Prefill partials [token * Hq + head][piece] behind the verify part's
// workspace; none when the chunks' keys are not split.
size_t prefill_partial_bytes(const pa_dims* d, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(d->total_tokens) * d->num_q_heads * splits;
  return align256(rows * d->head_dim * 4) + 2 * align256(rows * 4);
}

size_t mixed_workspace_bytes(const pa_dims* d, const pa_plan& plan, int32_t max_ctx, int32_t window, pa_dtype kv,
                             int sms) {
  const int splits = kv == PA_F32 ? 1 : prefill_geometry(d, max_ctx, window, sms).splits;  // fp32: one pass
  return workspace_bytes_for(d, plan, true) + prefill_partial_bytes(d, splits);
}

int device_sm_count(int* out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *out = v;
      return PA_OK;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return PA_ERR_CUDA;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA descriptor over one cache: dims {D, ps, Hkv, num_blocks}, box
// {128 bytes of a row, box_rows slots, 1 head, 1 page}, 128-byte swizzle.
int encode_cache_map(CUtensorMap* m, const void* base, pa_dtype kv, const pa_dims* d, int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PA_ERR_CUDA;
  const int eb = dtype_bytes(kv);
  const cuuint64_t D = d->head_dim, ps = d->page_size;
  const cuuint64_t head_stride = (kv == PA_U8) ? ps * (D + 4) : ps * D * eb;
  cuuint64_t dims[4] = {D, ps, static_cast<cuuint64_t>(d->num_kv_heads), static_cast<cuuint64_t>(d->num_blocks)};
  cuuint64_t strides[3] = {D * eb, head_stride, head_stride * d->num_kv_heads};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = kv == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                : kv == PA_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = enc(m, t, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// TMA descriptor over a u8 cache's page-head records viewed as 64-byte rows:
// dims {64, record / 64, Hkv, num_blocks}, one box = one whole record (codes,
// scales, zero-points), 64-byte swizzle.
int encode_u8_record_map(CUtensorMap* m, const void* base, const pa_dims* d) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PA_ERR_CUDA;
  const cuuint64_t rec = static_cast<cuuint64_t>(d->page_size) * (d->head_dim + 4);
  if (rec % 64 != 0 || rec / 64 > 256) return PA_ERR_UNSUPPORTED;
  cuuint64_t dims[4] = {64, rec / 64, static_cast<cuuint64_t>(d->num_kv_heads), static_cast<cuuint64_t>(d->num_blocks)};
  cuuint64_t strides[3] = {64, rec, rec * d->num_kv_heads};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rec / 64), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// TMA descriptor over a u8 V cache for the warp-level kernel: the codes of a
// page-head record are dim-major, viewed as dims {ps (keys), D (head dims),
// Hkv, num_blocks}; one box = box_rows keys of every head dim, no swizzle.
int encode_u8_v_map(CUtensorMap* m, const void* base, const pa_dims* d, int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PA_ERR_CUDA;
  const cuuint64_t ps = d->page_size, D = d->head_dim;
  const cuuint64_t rec = ps * (D + 4);
  cuuint64_t dims[4] = {ps, D, static_cast<cuuint64_t>(d->num_kv_heads), static_cast<cuuint64_t>(d->num_blocks)};
  cuuint64_t strides[3] = {ps, rec, rec * d->num_kv_heads};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(D), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

struct Call {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* bt;
  const int32_t* past_lens;
  const int32_t* begins;
  int32_t max_ctx;
  float scale;
  int32_t window;
  pa_dtype kv;
  void* out;
  const pa_dims* d;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  int32_t* trace;
  const uint8_t* tree_mask = nullptr;  // optional (tree-mask verify)
  int role = pa::kRoleAll;             // which sequences the launches serve
  bool clear_status = false;           // zero the status word on the stream just before the launches
};

PartArgs part_args(const Call& c, const pa_plan& plan, const Workspace& w) {
  const pa_dims* d = c.d;
  PartArgs a;
  a.q = c.q;
  a.k_bytes = static_cast<const uint8_t*>(c.k);
  a.v_bytes = static_cast<const uint8_t*>(c.v);
  a.block_tables = c.bt;
  a.past_lens = c.past_lens;
  a.begins = c.begins;
  a.out = c.out;
  a.po = w.po;
  a.pm = w.pm;
  a.pl = w.pl;
  a.status = w.status;
  a.trace = c.trace;
  a.tree_mask = c.tree_mask;
  a.num_seqs = d->num_seqs;
  a.total_tokens = d->total_tokens;
  a.Hq = d->num_q_heads;
  a.Hkv = d->num_kv_heads;
  a.G = d->num_q_heads / d->num_kv_heads;
  a.D = d->head_dim;
  a.ps = d->page_size;
  a.ps_log2 = ilog2(d->page_size);
  a.num_blocks = d->num_blocks;
  a.max_blocks = d->max_blocks_per_seq;
  a.max_ctx = c.max_ctx;
  a.window = c.window;
  a.part_tokens = plan.part_tokens;
  a.num_parts = plan.num_partitions;
  a.box_log2 = ilog2(std::min(d->page_size, plan.stage_keys));
  a.row_cap = plan.kernel == 0   ? pa::kConsumerWarps * 8 * plan.row_tiles
              : plan.kernel == 2 ? 64
              : plan.kernel == 4 ? plan.row_tiles
                                 : (1 << 30);
  a.q_dtype = d->q_dtype;
  a.out_dtype = d->out_dtype;
  a.scale_log2 = c.scale * 1.4426950408889634f;
  a.role = c.role;
  a.num_sms = plan.num_sms;
  return a;
}

int launch_partition(const Call& c, const pa_plan& plan, const Workspace& w) {
  const pa_dims* d = c.d;
  const PartArgs a = part_args(c, plan, w);
  const int box_rows = std::min(d->page_size, plan.stage_keys);
  const dim3 grid(plan.num_partitions, d->num_kv_heads, d->num_seqs);

  cudaError_t e;
  if (plan.kernel == 4) {
    CUtensorMap mk;
    const int rc = encode_u8_record_map(&mk, c.k, d);
    if (rc != PA_OK) return rc;
    e = pa::launch_u8(plan.row_tiles, d->page_size, mk, a, grid, c.stream);
  } else if (plan.kernel == 2 && d->page_size < pa::kGatherBelowPageSize) {
    e = pa::launch_tc_gather(d->head_dim, mma_kind(c.kv), a, grid, c.stream);
  } else if (plan.kernel == 2) {
    CUtensorMap mk, mv;
    int rc = encode_cache_map(&mk, c.k, c.kv, d, box_rows);
    if (rc == PA_OK) rc = encode_cache_map(&mv, c.v, c.kv, d, box_rows);
    if (rc != PA_OK) return rc;
    e = pa::launch_tc(d->head_dim, mma_kind(c.kv), mk, mv, a, grid, c.stream);
  } else if (plan.kernel == 0 && d->page_size < pa::kGatherBelowPageSize) {
    e = pa::launch_mma_d256_gather(mma_kind(c.kv), a, grid, c.stream);
  } else if (plan.kernel == 0) {
    CUtensorMap mk, mv;
    int rc = encode_cache_map(&mk, c.k, c.kv, d, box_rows);
    if (rc == PA_OK)
      rc = c.kv == PA_U8 ? encode_u8_v_map(&mv, c.v, d, box_rows) : encode_cache_map(&mv, c.v, c.kv, d, box_rows);
    if (rc != PA_OK) return rc;
    const int kind = mma_kind(c.kv);
    if (d->head_dim == 64) e = pa::launch_mma_d64(kind, plan.row_tiles, mk, mv, a, grid, c.stream);
    else if (d->head_dim == 128) e = pa::launch_mma_d128(kind, plan.row_tiles, mk, mv, a, grid, c.stream);
    else e = pa::launch_mma_d256(kind, plan.row_tiles, mk, mv, a, grid, c.stream);
  } else {
    if (d->head_dim == 64) e = pa::launch_dependent(pa::pa_partition_f32<64>, grid, dim3(128), 0, c.stream, a);
    else if (d->head_dim == 128) e = pa::launch_dependent(pa::pa_partition_f32<128>, grid, dim3(128), 0, c.stream, a);
    else e = pa::launch_dependent(pa::pa_partition_f32<256>, grid, dim3(128), 0, c.stream, a);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int launch_combine(const Call& c, const pa_plan& plan, const Workspace& w) {
  const pa_dims* d = c.d;
  if (plan.num_partitions <= 1) return PA_OK;  // every sequence was written directly
  CombineArgs a;
  a.past_lens = c.past_lens;
  a.begins = c.begins;
  a.out = c.out;
  a.po = w.po;
  a.pm = w.pm;
  a.pl = w.pl;
  a.status = w.status;
  a.num_seqs = d->num_seqs;
  a.total_tokens = d->total_tokens;
  a.Hq = d->num_q_heads;
  a.Hkv = d->num_kv_heads;
  a.G = d->num_q_heads / d->num_kv_heads;
  a.ps = d->page_size;
  a.max_ctx = c.max_ctx;
  a.window = c.window;
  a.part_tokens = plan.part_tokens;
  a.num_parts = plan.num_partitions;
  a.row_cap = plan.kernel == 0   ? pa::kConsumerWarps * 8 * plan.row_tiles
              : plan.kernel == 2 ? 64
              : plan.kernel == 4 ? plan.row_tiles
                                 : (1 << 30);
  a.out_dtype = d->out_dtype;
  a.role = c.role;
  a.num_sms = plan.num_sms;
  const long long rows = static_cast<long long>(d->total_tokens) * d->num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + pa::kCombineRows - 1) / pa::kCombineRows));
  cfg.blockDim = dim3(pa::kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (d->head_dim == 64) e = cudaLaunchKernelEx(&cfg, pa::pa_combine<64>, a);
  else if (d->head_dim == 128) e = cudaLaunchKernelEx(&cfg, pa::pa_combine<128>, a);
  else e = cudaLaunchKernelEx(&cfg, pa::pa_combine<256>, a);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int check_pointers(const Call& c, bool need_tensors, bool need_workspace = true) {
  if (c.begins == nullptr || c.past_lens == nullptr || c.out == nullptr) return PA_ERR_NULL;
  if (need_workspace && c.ws == nullptr) return PA_ERR_NULL;
  if (need_tensors && (c.q == nullptr || c.k == nullptr || c.v == nullptr || c.bt == nullptr)) return PA_ERR_NULL;
  if (!aligned(c.out, 16) || (need_workspace && !aligned(c.ws, 16)) || !aligned(c.begins, 4) ||
      !aligned(c.past_lens, 4))
    return PA_ERR_ALIGN;
  if (need_tensors && (!aligned(c.q, 16) || !aligned(c.k, 16) || !aligned(c.v, 16) || !aligned(c.bt, 4)))
    return PA_ERR_ALIGN;
  if (c.trace != nullptr && !aligned(c.trace, 4)) return PA_ERR_ALIGN;
  return PA_OK;
}

int run(const Call& c, bool do_partition, bool do_combine) {
  if (c.d == nullptr) return PA_ERR_NULL;
  int sms = 0;
  pa_plan plan;
  int rc = make_plan(c.d, c.max_ctx, c.window, c.kv, 1, &plan);  // argument checks first
  if (rc != PA_OK) return rc;
  rc = check_pointers(c, do_partition);
  if (rc != PA_OK) return rc;
  if (c.d->total_tokens == 0) return PA_OK;
  rc = device_sm_count(&sms);
  if (rc != PA_OK) return rc;
  rc = make_plan(c.d, c.max_ctx, c.window, c.kv, sms, &plan);
  if (rc != PA_OK) return rc;
  if (c.ws_bytes < workspace_bytes_for(c.d, plan)) return PA_ERR_WORKSPACE;
  const Workspace w = carve(c.ws, c.d, plan);
  // every check has passed: from here on the call enqueues work
  if (c.clear_status && cudaMemsetAsync(w.status, 0, sizeof(uint32_t), c.stream) != cudaSuccess) return PA_ERR_CUDA;
  if (do_partition) {
    rc = launch_partition(c, plan, w);
    if (rc != PA_OK) return rc;
  }
  if (do_combine) rc = launch_combine(c, plan, w);
  return rc;
}

// The prefill chunks (T_b > 8) of a mixed call: 128-row tiles on the
// tensor cores (16-bit caches), or the FFMA kernel with one partition per
// sequence (fp32 caches).  Outputs are written directly.
int launch_prefill(const Call& c, const pa_plan& plan, const Workspace& w) {
  const pa_dims* d = c.d;
  PartArgs a = part_args(c, plan, w);
  a.role = pa::kRoleLong;
  a.tree_mask = nullptr;  // prefill chunks follow the causal chain
  cudaError_t e;
  if (c.kv == PA_F32) {
    a.part_tokens = 1 << 30;  // one partition: the output row directly
    a.num_parts = 1;
    const dim3 grid(1, d->num_kv_heads, d->num_seqs);
    if (d->head_dim == 64) e = pa::launch_dependent(pa::pa_partition_f32<64>, grid, dim3(128), 0, c.stream, a);
    else if (d->head_dim == 128) e = pa::launch_dependent(pa::pa_partition_f32<128>, grid, dim3(128), 0, c.stream, a);
    else e = pa::launch_dependent(pa::pa_partition_f32<256>, grid, dim3(128), 0, c.stream, a);
  } else {
    int sms = 0;
    if (device_sm_count(&sms) != PA_OK) return PA_ERR_CUDA;
    const PrefillGeometry pg = prefill_geometry(d, c.max_ctx, c.window, sms);
    a.row_cap = pg.rows_per_block;
    if (pg.tiles > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (pg.tiles == 0) return PA_OK;
    if (pg.splits > 1) {
      // the pieces' partial rows, after the verify part's workspace
      const size_t rows = static_cast<size_t>(d->total_tokens) * d->num_q_heads * pg.splits;
      uint8_t* base = reinterpret_cast<uint8_t*>(w.status) + workspace_bytes_for(d, plan, true);
      a.po = reinterpret_cast<float*>(base);
      a.pm = reinterpret_cast<float*>(base + align256(rows * d->head_dim * 4));
      a.pl = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.pm) + align256(rows * 4));
      a.num_parts = pg.splits;
    }
    const int box_rows = std::min(d->page_size, 64);
    a.box_log2 = ilog2(box_rows);
    CUtensorMap mk, mv;
    int rc = encode_cache_map(&mk, c.k, c.kv, d, box_rows);
    if (rc == PA_OK) rc = encode_cache_map(&mv, c.v, c.kv, d, box_rows);
    if (rc != PA_OK) return rc;
    e = pa::launch_prefill_tc(d->head_dim, mma_kind(c.kv), mk, mv, a,
                              dim3(static_cast<unsigned>(pg.tiles), d->num_kv_heads, pg.splits), c.stream);
    if (e == cudaSuccess && pg.splits > 1) {
      CombineArgs ca;
      ca.past_lens = c.past_lens;
      ca.begins = c.begins;
      ca.out = c.out;
      ca.po = a.po;
      ca.pm = a.pm;
      ca.pl = a.pl;
      ca.status = w.status;
      ca.num_seqs = d->num_seqs;
      ca.total_tokens = d->total_tokens;
      ca.Hq = d->num_q_heads;
      ca.Hkv = d->num_kv_heads;
      ca.G = d->num_q_heads / d->num_kv_heads;
      ca.ps = d->page_size;
      ca.max_ctx = c.max_ctx;
      ca.window = c.window;
      ca.part_tokens = a.part_tokens;
      ca.num_parts = pg.splits;
      ca.row_cap = pg.rows_per_block;
      ca.out_dtype = d->out_dtype;
      ca.role = pa::kRoleLong;
      ca.num_sms = sms;
      e = pa::launch_prefill_combine(d->head_dim, ca, c.stream);
    }
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Argument checks of a mixed call beyond the verify part's plan.
int mixed_support(const pa_dims* d, pa_dtype kv) {
  const bool tc16 = (kv == PA_BF16 || kv == PA_F16) && d->head_dim <= 128;
  if (kv != PA_F32 && !tc16) return PA_ERR_UNSUPPORTED;
  if (tc16 && d->page_size < pa::kGatherBelowPageSize) return PA_ERR_PAGE_SIZE;
  if (tc16 && d->num_q_heads / d->num_kv_heads > 128) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

int run_mixed(Call c) {
  if (c.d == nullptr) return PA_ERR_NULL;
  pa_plan plan;
  int rc = make_plan(c.d, c.max_ctx, c.window, c.kv, 1, &plan);
  if (rc != PA_OK) return rc;
  rc = mixed_support(c.d, c.kv);
  if (rc != PA_OK) return rc;
  rc = check_pointers(c, true);
  if (rc != PA_OK) return rc;
  if (c.d->total_tokens == 0) return PA_OK;
  int sms = 0;
  rc = device_sm_count(&sms);
  if (rc != PA_OK) return rc;
  rc = make_plan(c.d, c.max_ctx, c.window, c.kv, sms, &plan);
  if (rc != PA_OK) return rc;
  if (c.ws_bytes < mixed_workspace_bytes(c.d, plan, c.max_ctx, c.window, c.kv, sms)) return PA_ERR_WORKSPACE;
  const Workspace w = carve(c.ws, c.d, plan, true);
  c.role = pa::kRoleShort;  // verify steps: split-KV partitions + combine
  rc = launch_partition(c, plan, w);
  if (rc == PA_OK) rc = launch_combine(c, plan, w);
  if (rc == PA_OK) rc = launch_prefill(c, plan, w);  // prefill chunks, after the combine in stream order
  return rc;
}

// ---------------------------------------------------------------------------
// Scratch for pa_verify_forward_no_alloc: a fixed device array that the
// library owns, so the caller needs no allocator.  Every GPU that loads the
// library holds these 16 MiB until the process exits.  All calls share it.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

// Device address of g_no_alloc_scratch in the current context.  In host code
// the array's name is only a host-side stand-in; kernels must be given this
// address.  It is resolved (cudaGetSymbolAddress, with the device current)
// the first time a context calls, and cached per device together with the
// context's unique id: a context made after a device reset (where the
// library's module, and so the array, may sit elsewhere) resolves it again.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the calling thread's current context (0 if none or unknown).
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int no_alloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static unsigned long long ctx_of[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    addr[dev] = p;
    ctx_of[dev] = current_context_id();  // the symbol lookup made the device's context current
  }
  *ptr = addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_verify_workspace_size(const pa_dims* dims, int32_t max_context_len, int32_t sliding_window,
                                pa_dtype kv_dtype) {
  int sms = 0;
  if (device_sm_count(&sms) != PA_OK) return 0;
  pa_plan plan;
  if (make_plan(dims, max_context_len, sliding_window, kv_dtype, sms, &plan) != PA_OK) return 0;
  // tree-mask calls run the same kernels with the same plan: one size serves both
  return workspace_bytes_for(dims, plan);
}

size_t pa_mixed_workspace_size(const pa_dims* dims, int32_t max_context_len, int32_t sliding_window,
                               pa_dtype kv_dtype) {
  int sms = 0;
  if (device_sm_count(&sms) != PA_OK) return 0;
  pa_plan plan;
  if (make_plan(dims, max_context_len, sliding_window, kv_dtype, sms, &plan) != PA_OK) return 0;
  if (mixed_support(dims, kv_dtype) != PA_OK) return 0;
  return mixed_workspace_bytes(dims, plan, max_context_len, sliding_window, kv_dtype, sms);
}

int pa_forward_mixed(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                     const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                     float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                     void* workspace, size_t workspace_bytes, void* cuda_stream) {
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr};
  return run_mixed(c);
}

int pa_forward_mixed_tree(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                          float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                          void* workspace, size_t workspace_bytes, const uint8_t* tree_mask, void* cuda_stream) {
  if (tree_mask == nullptr) return PA_ERR_NULL;
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr, tree_mask};
  return run_mixed(c);
}

int pa_verify_plan(const pa_dims* dims, int32_t max_context_len, int32_t sliding_window, pa_dtype kv_dtype,
                   int32_t num_sms, pa_plan* plan) {
  return make_plan(dims, max_context_len, sliding_window, kv_dtype, num_sms, plan);
}

int pa_verify_forward(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                      float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                      void* workspace, size_t workspace_bytes, void* cuda_stream) {
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr};
  return run(c, true, true);
}

int pa_verify_forward_tree(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                           float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                           void* workspace, size_t workspace_bytes, const uint8_t* tree_mask, void* cuda_stream) {
  if (tree_mask == nullptr) return PA_ERR_NULL;
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr, tree_mask};
  return run(c, true, true);
}

int pa_verify_forward_traced(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                             const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                             float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                             void* workspace, size_t workspace_bytes, void* cuda_stream, int32_t* gather_trace) {
  if (gather_trace == nullptr) return PA_ERR_NULL;
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), gather_trace};
  return run(c, true, true);
}

int pa_verify_partition(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                        float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                        void* workspace, size_t workspace_bytes, void* cuda_stream) {
  const Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
               max_context_len, scale, sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr};
  return run(c, true, false);
}

int pa_verify_combine(const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                      int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims, void* workspace,
                      size_t workspace_bytes, void* cuda_stream) {
  const Call c{nullptr, nullptr, nullptr, nullptr, past_lens, subsequence_begins, max_context_len, 1.0f,
               sliding_window, kv_dtype, out, dims, workspace, workspace_bytes,
               static_cast<cudaStream_t>(cuda_stream), nullptr};
  return run(c, false, true);
}

int pa_verify_forward_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* past_lens,
                               const int32_t* subsequence_begins, int32_t max_context_len, float scale,
                               int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                               void* cuda_stream) {
  if (dims == nullptr) return PA_ERR_NULL;
  Call c{q,     k_cache,        v_cache, block_tables, past_lens, subsequence_begins,
         max_context_len, scale, sliding_window, kv_dtype, out, dims, nullptr, kNoAllocScratchBytes,
         static_cast<cudaStream_t>(cuda_stream), nullptr};
  // Host-only checks first, so that a rejected call makes no CUDA call and
  // enqueues nothing.
  pa_plan plan;
  int rc = make_plan(dims, max_context_len, sliding_window, kv_dtype, 1, &plan);
  if (rc != PA_OK) return rc;
  rc = check_pointers(c, true, false);
  if (rc != PA_OK) return rc;
  if (dims->total_tokens == 0) return PA_OK;
  void* scratch = nullptr;
  rc = no_alloc_scratch(&scratch);
  if (rc != PA_OK) return rc;
  c.ws = scratch;
  // The status word is the only part of the scratch that must start at zero
  // (partials are written before they are read); run() clears it on the
  // stream once the plan and the size check have passed.
  c.clear_status = true;
  return run(c, true, true);  // PA_ERR_WORKSPACE when the call needs more than the scratch holds
}

int pa_verify_get_device_status(void* workspace, void* cuda_stream, uint32_t* bits) {
  if (workspace == nullptr || bits == nullptr) return PA_ERR_NULL;
  if (!aligned(workspace, 16)) return PA_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  *bits = host;
  return PA_OK;
}

const char* pa_verify_status_string(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_DTYPE: return "unsupported q / kv / out dtype combination";
    case PA_ERR_SHAPE: return "invalid dimensions";
    case PA_ERR_HEAD_DIM: return "unsupported head_dim";
    case PA_ERR_PAGE_SIZE: return "unsupported page_size";
    case PA_ERR_ALIGN: return "misaligned pointer";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CONTEXT: return "max_context_len out of range";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_UNSUPPORTED: return "query rows per KV head exceed the supported maximum";
    default: return "unknown status code";
  }
}

}  // extern "C"
