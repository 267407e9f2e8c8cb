// pa_device.cuh — device-side building blocks of the paged verify-attention
// kernels for sm_103a: mbarrier / TMA / bulk-copy wrappers, warp-level mma
// fragments, and the per-sequence bookkeeping shared by the partition and
// combine kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <climits>

#include "../../include/pa_verify.h"

namespace pa {

enum KvKind : int { KV_BF16 = 0, KV_F16 = 1, KV_U8 = 2 };

constexpr int kConsumerWarps = 4;            // warps that do the math
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one TMA producer warp
constexpr int kMaxPagesPerCta = 1024;        // block ids staged in shared memory
constexpr int kGatherWarps = 4;              // cp.async producer warps of the small-page gather
constexpr uint32_t kWaitLimit = 1u << 22;    // bounded mbarrier polls before giving up

// Arguments common to the partition kernels (plain values, passed by value).
// Which sequences a launch serves.  A plain verify call serves all of them
// (T_b <= 8).  A mixed call runs the split-KV kernels over its verify steps
// (T_b <= 8; their partials indexed by slot b * 8 + i, so the workspace does
// not grow with prefill tokens) and the prefill kernel over its prefill
// chunks (T_b > 8).
constexpr int kRoleAll = 0, kRoleShort = 1, kRoleLong = 2;

struct PartArgs {
  const void* q;
  const uint8_t* k_bytes;       // cache bases (u8 records need byte addressing)
  const uint8_t* v_bytes;
  const int32_t* block_tables;
  const int32_t* past_lens;
  const int32_t* begins;
  void* out;
  float* po;                    // [slots, Hq, P, D] unnormalised partial outputs
  float* pm;                    // [slots, Hq, P] running max (log2 domain)
  float* pl;                    // [slots, Hq, P] softmax denominators (-1 = poisoned)
                                // slots: total_tokens (token t), or B * 8 in a
                                // mixed call's verify part (b * 8 + i)
  uint32_t* status;
  int32_t* trace;               // optional gather trace
  const uint8_t* tree_mask;     // optional: per token, bit k = sees new token k of its sequence
  int num_seqs, total_tokens, Hq, Hkv, G, D, ps, ps_log2, num_blocks, max_blocks;
  int max_ctx, window, part_tokens, num_parts, box_log2, row_cap;
  int q_dtype, out_dtype;
  int role;                     // kRoleAll / kRoleShort / kRoleLong
  int num_sms;                  // SMs of the device (prefill key pieces)
  float scale_log2;             // softmax scale * log2(e)
};

struct CombineArgs {
  const int32_t* past_lens;
  const int32_t* begins;
  void* out;
  const float* po;
  const float* pm;
  const float* pl;
  uint32_t* status;
  int num_seqs, total_tokens, Hq, Hkv, G, ps, max_ctx, window, part_tokens, num_parts, row_cap, out_dtype;
  int role;
  int num_sms;
};

// ---------------------------------------------------------------------------
// Per-sequence bookkeeping (identical in the partition and combine kernels).
// ---------------------------------------------------------------------------
struct SeqInfo {
  int t0, T, L;          // first token row, new tokens, past length
  int klo, khi;          // union of the rows' key ranges [klo, khi]
  int kbase;             // klo rounded down to a page boundary
  int nparts;            // partitions this sequence needs
  long long pshift;      // partials of token t live at token slot t + pshift (prow)
  bool foreign;          // another kernel of a mixed call owns this sequence
  uint32_t err;          // PA_STATUS_* bits that make the sequence invalid
  bool rows_ok;          // t0 / T can be trusted to index output rows
};

// A global load the compiler issues exactly once: a read-only (__ldg) load
// may legally be repeated at each use instead of holding the value in a
// register, and under a saturated memory system every repeat costs a full
// round trip.
__device__ __forceinline__ int32_t ld_once(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_once_u8(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
// The new tokens token i of a sequence sees: its tree mask, or the causal
// chain 0..i when there is none.
__device__ __forceinline__ uint32_t row_new_token_mask(const uint8_t* tree_mask, int t, int i) {
  return tree_mask != nullptr ? ld_once_u8(tree_mask + t) : ((2u << i) - 1u);
}
__device__ __forceinline__ uint32_t ld_once(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ SeqInfo seq_info(const int32_t* begins, const int32_t* past_lens, int b,
                                            int total_tokens, int G, int ps, int max_ctx, int window,
                                            int part_tokens, int row_capacity, int role) {
  SeqInfo s;
  s.t0 = ld_once(begins + b);
  const int t1 = ld_once(begins + b + 1);
  s.L = ld_once(past_lens + b);
  s.T = t1 - s.t0;
  s.err = 0;
  s.pshift = role == kRoleShort ? static_cast<long long>(b) * PA_MAX_QUERY_LEN - s.t0 : 0;
  s.foreign = false;
  s.rows_ok = (s.t0 >= 0 && t1 >= s.t0 && t1 <= total_tokens);
  // a mixed call splits its sequences by length: verify steps (T <= 8) to
  // the split-KV kernels, prefill chunks (T > 8) to the prefill kernel
  if (s.rows_ok && ((role == kRoleShort && s.T > PA_MAX_QUERY_LEN) || (role == kRoleLong && s.T <= PA_MAX_QUERY_LEN))) {
    s.foreign = true;
    s.T = 0;
  }
  if (!s.rows_ok) s.err |= PA_STATUS_BEGINS;
  if (role != kRoleLong && s.T > PA_MAX_QUERY_LEN) s.err |= PA_STATUS_QUERY_LEN;
  if (s.L < 0) s.err |= PA_STATUS_PAST_LEN;
  if ((long long)s.L + s.T > (long long)max_ctx) s.err |= PA_STATUS_CONTEXT;
  if (role != kRoleLong && s.T * G > row_capacity) s.err |= PA_STATUS_ROWS;
  s.khi = s.L + s.T - 1;
  s.klo = window > 0 ? max(0, s.L - window + 1) : 0;
  s.kbase = (s.klo / ps) * ps;
  s.nparts = (s.err || s.T <= 0) ? 0 : (s.khi + 1 - s.kbase + part_tokens - 1) / part_tokens;
  return s;
}

// Fewest keys a prefill block's key piece takes: a block with fewer keys than
// pieces x this uses fewer pieces (prefill_block_pieces).
constexpr int kPrefillMinPieceKeys = 4096;

__device__ __forceinline__ int prefill_block_pieces(int pieces, int keys) {
  return max(1, min(pieces, keys / kPrefillMinPieceKeys));
}

// Key pieces of a mixed call's prefill blocks, from the blocks the batch
// really has (sequences with T_b > 8, TQ tokens per block): as many as fit in
// one wave of the SMs, at most `max_pieces` (the launch's grid.z and the
// partial rows' stride).  Warp-collective: every lane returns the count.
__device__ __forceinline__ int prefill_pieces(const int32_t* begins, int num_seqs, int TQ, int Hkv, int max_pieces,
                                              int num_sms) {
  if (max_pieces <= 1) return 1;
  const int lane = threadIdx.x & 31;
  long long blocks = 0;
  for (int s = lane; s < num_seqs; s += 32) {
    const int T = ld_once(begins + s + 1) - ld_once(begins + s);
    if (T > PA_MAX_QUERY_LEN) blocks += (T + TQ - 1) / TQ;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) blocks += __shfl_xor_sync(0xffffffffu, blocks, off);
  const long long ctas = blocks * Hkv;
  if (ctas <= 0) return 1;
  return static_cast<int>(max(1LL, min(static_cast<long long>(max_pieces), num_sms / ctas)));
}

// Partial-buffer row of output row `row` (= t * Hq + h) of a sequence.
__device__ __forceinline__ size_t prow(size_t row, const SeqInfo& si, int Hq) {
  return static_cast<size_t>(static_cast<long long>(row) + si.pshift * Hq);
}

// ---------------------------------------------------------------------------
// Small numeric helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// c + a * b with f16 a, b and f32 c: the product is exact in f32 and the sum
// is rounded once, as fmaf on the widened operands would, without widening.
__device__ __forceinline__ float fma_f16_f32(uint16_t a_bits, uint16_t b_bits, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a_bits), "h"(b_bits), "f"(c));
  return d;
}

// Reduces each of a lane's NV values (NV a power of two, <= 32) over the
// warp's 32 lanes by recursive halving: at each exchange a lane keeps one half
// of its values, sends the other half to its partner and combines what comes
// back, so the warp spends NV - 1 + log2(32 / NV) shuffles instead of 5 NV.
// v is overwritten.  Returns, in lane l, the reduction of value l / (32 / NV).
template <int NV, typename Op>
__device__ __forceinline__ float warp_reduce_split(float* v, int lane, Op op) {
  static_assert(NV >= 1 && NV <= 32 && (NV & (NV - 1)) == 0, "NV: a power of two up to 32");
  int o = 16;
#pragma unroll
  for (int n = NV; n > 1; n >>= 1) {
    const bool up = (lane & o) != 0;  // this lane keeps the upper half
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
    o >>= 1;
  }
  float t = v[0];
#pragma unroll
  for (int k = 32 / NV / 2; k > 0; k >>= 1) t = op(t, __shfl_xor_sync(0xffffffffu, t, k));
  return t;
}
struct OpAdd {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};
struct OpMax {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};

__device__ __forceinline__ float load_q_elem(const void* q, int dtype, size_t idx) {
  if (dtype == PA_F32) return __ldg(reinterpret_cast<const float*>(q) + idx);
  const unsigned short bits = __ldg(reinterpret_cast<const unsigned short*>(q) + idx);
  if (dtype == PA_BF16) return __bfloat162float(__ushort_as_bfloat16(bits));
  return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ void store_out(void* out, int dtype, size_t idx, float v) {
  if (dtype == PA_F32) {
    reinterpret_cast<float*>(out)[idx] = v;
  } else if (dtype == PA_BF16) {
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

// Four consecutive output elements (idx a multiple of 4), packed as the output
// type: one 16-byte (fp32) or 8-byte (16-bit) store.
__device__ __forceinline__ void store_out4(void* out, int dtype, size_t idx, float4 v) {
  if (dtype == PA_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx) = v;
  } else if (dtype == PA_BF16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  } else {
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(out) + idx) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and asynchronous copies (PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking probe of a phase (for issuers that poll several barriers).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: true when the phase completed, false after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Pull a tensor map into the descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Barrier-reduction over the `n` threads of named barrier `id`: true when the
// predicate holds on any of them (all of them wait for each other).
__device__ __forceinline__ bool bar_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_sync_n(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// L2 prefetches: a hint only, nothing returns to the program.  Issued before
// griddepcontrol.wait they warm L2 with lines the kernel will read once the
// previous kernel is done; a later write by that kernel updates the line.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}
// bytes: a multiple of 16, src 16-byte aligned.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// 4-byte asynchronous global -> shared copy (completion: cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// 16-byte asynchronous global -> shared copy; src_bytes = 0 reads nothing and
// writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on an mbarrier once this thread's earlier cp.async copies have
// landed; .noinc: the barrier's expected count already includes the arrival.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier among the consumer warps only (the producer warp skips it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (mma.sync m16n8k16, fp32 accumulate).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (kBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Transpose an 8x8 16-bit matrix held in mma fragment layout across the warp.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Two u8 codes (bytes sel0 / sel1 of w) -> exact f16x2: place each byte in
// the mantissa of 1024.0 (0x6400) and subtract 1024.
__device__ __forceinline__ uint32_t u8pair_to_f16x2(uint32_t w, uint32_t selector) {
  uint32_t h = __byte_perm(w, 0x64646464u, selector);
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&h), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Row permutation of the 16 keys of an mma tile: m -> key offset.  Pairs of
// keys read by one quarter-warp land in different shared-memory bank halves
// under the 128-byte swizzle (see the u8 fragment loaders).
__device__ __forceinline__ int key_perm(int m) { return (m & 8) | ((5 * m) & 7); }

// Byte offset of (key k of the stage, 128-byte column chunk c) in a stage tile
// laid out as [segment][chunk][box_rows][128 B], box_rows = 1 << box_log2.
__device__ __forceinline__ uint32_t tile_row_off(int k, int c, int box_log2, int n_chunks) {
  const int br = 1 << box_log2;
  return static_cast<uint32_t>((((k >> box_log2) * n_chunks + c) * br + (k & (br - 1))) * 128);
}

// 128-byte swizzle: 16-byte unit j of the row of key k sits at unit j ^ (k & 7).
__device__ __forceinline__ uint32_t swz(int unit, int k) { return static_cast<uint32_t>(((unit ^ (k & 7)) << 4)); }

}  // namespace pa
