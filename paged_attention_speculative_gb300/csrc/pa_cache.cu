// pa_cache.cu — the cache update: the step just before the verify, which
// writes the T new tokens' K and V into their pages (the OpenVINO
// paged-attention op stores the new tokens itself, issue 38153 reproduction
// step 3; u8 KV cache precision, step 1).
//
// Token i of sequence b goes to position p = past_len_b + i: page
// block_tables[b][p / ps], slot p % ps, for every KV head, K and V alike.
// Float caches store the value rounded to nearest-even in the cache dtype.
// u8 caches get one scale / zero-point pair per token and KV head, computed
// in binary32 with every operation rounded to nearest-even (the integer
// codes depend on it, so the steps are fixed):
//   mn = min x, mx = max x over the head's D values
//   scale = fp16((mx - mn) / 255)            1.0 if that is 0 or not finite
//   zp    = fp16((0 - mn) / scale)
//   code  = clamp(rint(x / scale + zp), 0, 255)
// One warp per (token, KV head, K-or-V); lane l owns D/32 consecutive values.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/pa_verify.h"
#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

struct CacheArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* block_tables;
  const int32_t* past_lens;
  const int32_t* begins;
  uint32_t* status;  // may be null
  int src_dtype, kv_dtype;
  int num_seqs, total_tokens, Hkv, ps, ps_log2, num_blocks, max_blocks;
};

template <int E>
__device__ __forceinline__ void load_src(const void* base, int dtype, size_t idx, float* x) {
  if (dtype == PA_F32) {
    const float* p = reinterpret_cast<const float*>(base) + idx;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 v = *reinterpret_cast<const float2*>(p + e);
      x[e] = v.x;
      x[e + 1] = v.y;
    }
  } else {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(base) + idx);
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const uint32_t w = p[e / 2];
      const float2 f = dtype == PA_BF16 ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w))
                                        : __half22float2(*reinterpret_cast<const __half2*>(&w));
      x[e] = f.x;
      x[e + 1] = f.y;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) pa_cache_update_kernel(const CacheArgs a) {
  constexpr int E = D / 32;  // values per lane
  pdl_wait_primary();        // the new K / V and the cache may belong to the previous kernel
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (item >= static_cast<long long>(a.total_tokens) * a.Hkv * 2) return;
  const int t = static_cast<int>(item / (2 * a.Hkv));
  const int rem = static_cast<int>(item % (2 * a.Hkv));
  const int g = rem >> 1;
  const bool is_v = (rem & 1) != 0;

  // the sequence of token t: the last b with begins[b] <= t
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ld_once(a.begins + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int t0 = ld_once(a.begins + lo), t1 = ld_once(a.begins + lo + 1);
  const int L = ld_once(a.past_lens + lo);
  uint32_t err = 0;
  if (!(t0 <= t && t < t1 && t1 <= a.total_tokens && ld_once(a.begins) == 0)) err |= PA_STATUS_BEGINS;
  if (L < 0) err |= PA_STATUS_PAST_LEN;
  const long long pos = static_cast<long long>(L) + (t - t0);
  const long long lp = pos >> a.ps_log2;
  int blk = 0;
  if (!err) {
    if (lp >= a.max_blocks) {
      err |= PA_STATUS_CONTEXT;
    } else {
      blk = ld_once(a.block_tables + static_cast<size_t>(lo) * a.max_blocks + lp);
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.num_blocks)) err |= PA_STATUS_BLOCK_ID;
    }
  }
  if (err) {  // the token's slot is not written
    if (lane == 0 && a.status != nullptr) atomicOr(a.status, err);
    return;
  }
  const int slot = static_cast<int>(pos & (a.ps - 1));

  float x[E];
  load_src<E>(is_v ? a.v_new : a.k_new, a.src_dtype, (static_cast<size_t>(t) * a.Hkv + g) * D + lane * E, x);
  void* cache = is_v ? a.v_cache : a.k_cache;

  if (a.kv_dtype != PA_U8) {
    const size_t base = ((static_cast<size_t>(blk) * a.Hkv + g) * a.ps + slot) * D + lane * E;
    if (a.kv_dtype == PA_F32) {
      float* dst = reinterpret_cast<float*>(cache) + base;
#pragma unroll
      for (int e = 0; e < E; e += 2) *reinterpret_cast<float2*>(dst + e) = make_float2(x[e], x[e + 1]);
    } else {
      uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(cache) + base);
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        uint32_t w;
        if (a.kv_dtype == PA_BF16) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(x[e], x[e + 1]);
          w = *reinterpret_cast<const uint32_t*>(&h);
        } else {
          const __half2 h = __floats2half2_rn(x[e], x[e + 1]);
          w = *reinterpret_cast<const uint32_t*>(&h);
        }
        dst[e / 2] = w;
      }
    }
    return;
  }

  // ---- u8: per-token scale / zero-point, then the codes ----
  if constexpr (E < 4) {
    return;  // u8 caches need head_dim 128 or 256 (rejected on the host)
  } else {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int e = 1; e < E; ++e) {
    mn = fminf(mn, x[e]);
    mx = fmaxf(mx, x[e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 255.0f));
  float sf = __half2float(s16);
  if (!(sf > 0.f) || isinf(sf)) {
    s16 = __ushort_as_half(0x3c00u);
    sf = 1.f;
  }
  const __half z16 = __float2half_rn(__fdiv_rn(__fsub_rn(0.f, mn), sf));
  const float zf = __half2float(z16);
  uint32_t packed[E / 4];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float c = rintf(__fadd_rn(__fdiv_rn(x[e], sf), zf));
    c = (c >= 0.f) ? fminf(c, 255.f) : 0.f;  // NaN -> 0 too
    const uint32_t b = static_cast<uint32_t>(c);
    if (e % 4 == 0) packed[e / 4] = b;
    else packed[e / 4] |= b << (8 * (e % 4));
  }
  uint8_t* rec = reinterpret_cast<uint8_t*>(cache) + (static_cast<size_t>(blk) * a.Hkv + g) * a.ps * (D + 4);
  if (!is_v) {
    // K records: codes slot-major, the token's D codes contiguous
    uint32_t* codes = reinterpret_cast<uint32_t*>(rec + static_cast<size_t>(slot) * D + lane * E);
#pragma unroll
    for (int w = 0; w < E / 4; ++w) codes[w] = packed[w];
  } else {
    // V records: codes dim-major, code of head dim d at d * ps + slot
#pragma unroll
    for (int e = 0; e < E; ++e)
      rec[static_cast<size_t>(lane * E + e) * a.ps + slot] = static_cast<uint8_t>(packed[e / 4] >> (8 * (e % 4)));
  }
  if (lane == 0) {
    *reinterpret_cast<__half*>(rec + static_cast<size_t>(a.ps) * D + 2 * slot) = s16;
    *reinterpret_cast<__half*>(rec + static_cast<size_t>(a.ps) * D + 2 * a.ps + 2 * slot) = z16;
  }
  }
}

}  // namespace pa

namespace {
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
int ilog2(int v) {
  int r = 0;
  while ((1 << r) < v) ++r;
  return r;
}
bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
}  // namespace

extern "C" int pa_cache_update(const void* k_new, const void* v_new, pa_dtype src_dtype, void* k_cache, void* v_cache,
                               pa_dtype kv_dtype, const int32_t* block_tables, const int32_t* past_lens,
                               const int32_t* subsequence_begins, const pa_dims* dims, uint32_t* status,
                               void* cuda_stream) {
  if (dims == nullptr) return PA_ERR_NULL;
  const pa_dims& d = *dims;
  if (d.num_seqs < 1 || d.total_tokens < 0 || d.num_kv_heads < 1 || d.num_blocks < 1 || d.max_blocks_per_seq < 1)
    return PA_ERR_SHAPE;
  const int D = d.head_dim;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_HEAD_DIM;
  if (!pow2(d.page_size) || d.page_size > 256) return PA_ERR_PAGE_SIZE;
  if (src_dtype != PA_F32 && src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_DTYPE;
  if (kv_dtype != PA_F32 && kv_dtype != PA_F16 && kv_dtype != PA_BF16 && kv_dtype != PA_U8) return PA_ERR_DTYPE;
  if (kv_dtype == PA_U8 && D == 64) return PA_ERR_HEAD_DIM;
  if (d.total_tokens == 0) return PA_OK;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr || block_tables == nullptr ||
      past_lens == nullptr || subsequence_begins == nullptr)
    return PA_ERR_NULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(past_lens, 4) || !aligned(subsequence_begins, 4) ||
      (status != nullptr && !aligned(status, 4)))
    return PA_ERR_ALIGN;
  pa::CacheArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.past_lens = past_lens;
  a.begins = subsequence_begins;
  a.status = status;
  a.src_dtype = src_dtype;
  a.kv_dtype = kv_dtype;
  a.num_seqs = d.num_seqs;
  a.total_tokens = d.total_tokens;
  a.Hkv = d.num_kv_heads;
  a.ps = d.page_size;
  a.ps_log2 = ilog2(d.page_size);
  a.num_blocks = d.num_blocks;
  a.max_blocks = d.max_blocks_per_seq;
  const long long items = static_cast<long long>(d.total_tokens) * d.num_kv_heads * 2;
  if ((items + 3) / 4 > 0x7fffffffLL) return PA_ERR_SHAPE;
  const dim3 grid(static_cast<unsigned>((items + 3) / 4));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e;
  if (D == 64) e = pa::launch_dependent(pa::pa_cache_update_kernel<64>, grid, dim3(128), 0, st, a);
  else if (D == 128) e = pa::launch_dependent(pa::pa_cache_update_kernel<128>, grid, dim3(128), 0, st, a);
  else e = pa::launch_dependent(pa::pa_cache_update_kernel<256>, grid, dim3(128), 0, st, a);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
