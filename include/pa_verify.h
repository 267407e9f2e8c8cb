/*
 * pa_verify.h — C ABI of the paged verify-attention library (libpa_verify.so).
 *
 * One call computes, for a batch of sequences that each bring T_b = 1..8 new
 * query tokens against a long paged KV cache, the attention output of every
 * new token, the way a speculative-decoding verify step needs it:
 *
 *   query token i of sequence b sits at position p = past_len_b + i and
 *   attends keys lo..p, lo = (W > 0) ? max(0, p - W + 1) : 0;
 *   out[t, h, :] = softmax_j(scale * q[t, h, :] . K_j) weighted sum of V_j,
 *   t = subsequence_begins[b] + i, with K_j / V_j of KV head h / (Hq / Hkv).
 *
 * Sources for the operation (web pages on paged attention in speculative
 * decoding):
 *  - OpenVINO issue 38153, "Performance issue description": a verify forward
 *    hands the paged-attention op k+1 query tokens of one sequence with a long
 *    past_len; the suggested handling gives query token i the key limit
 *    past_len + i + 1, equal to i single-token decodes.  "Cause": the fast
 *    single-token stage reads each KV head once for all GQA heads and splits
 *    the context into partitions — both kept here for T > 1.
 *  - OpenVINO issue 38153, "Step-by-step reproduction" step 3: the op inputs
 *    past_lens, subsequence_begins, max_context_len and the block table; step 1:
 *    u8 KV cache precision.
 *  - dual-radeon-vllm article (speculative decoding net loss), section on the
 *    use_3d gate: the split-KV segment buffer must be indexed per query token,
 *    not per sequence; a segment reduction merges the partial results.
 *  - SGLang discussion 36314, "Observation 3": sliding-window layers (window
 *    1024) read only the last window of keys.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers of the current CUDA device,
 *    owned by the caller.  The library allocates nothing, keeps no per-call
 *    state and never synchronises (except pa_verify_get_device_status, which
 *    synchronises the given stream).  All work is enqueued on `cuda_stream`
 *    (a cudaStream_t; NULL = legacy default stream).
 *  - q, k_cache, v_cache, out and workspace must be 16-byte aligned; the int32
 *    arrays 4-byte aligned.
 *  - Return value: PA_OK (0) or a negative PA_ERR_* code.  On a negative code
 *    nothing was enqueued (except PA_ERR_CUDA, which reports a failed launch).
 *  - Inconsistencies only visible on the device (a query length outside
 *    0..8, past_len + T_b > max_context_len, a block id outside
 *    [0, num_blocks), malformed subsequence_begins) set bits of a sticky
 *    status word inside the workspace (PA_STATUS_*), skip the affected work
 *    and leave the affected sequence's output rows zero.  Nothing traps.
 */
#ifndef PA_VERIFY_H
#define PA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  PA_U8 is valid only as a KV-cache type. */
typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_U8 = 3 } pa_dtype;

/* Host-detected errors (returned; nothing launched). */
enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer is NULL                          */
  PA_ERR_DTYPE = -2,       /* unsupported q / kv / out dtype combination          */
  PA_ERR_SHAPE = -3,       /* non-positive count, Hq % Hkv != 0, bad table width  */
  PA_ERR_HEAD_DIM = -4,    /* head_dim not in {64, 128, 256} (u8: {128, 256})     */
  PA_ERR_PAGE_SIZE = -5,   /* page_size not a power of two in [1, 256]; pages of
                              1, 2 or 4 tokens need an fp32 or a 16-bit cache
                              (head_dim <= 128: <= 64 query rows per KV head);
                              u8 caches need pages of 16 tokens or more
                              (pa_cache_update: any power of two up to 256)  */
  PA_ERR_ALIGN = -6,       /* a pointer misses its alignment                      */
  PA_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than pa_verify_workspace_size */
  PA_ERR_CONTEXT = -8,     /* max_context_len < 1 while tokens are present, or too large */
  PA_ERR_CUDA = -9,        /* a CUDA runtime call or kernel launch failed          */
  PA_ERR_UNSUPPORTED = -10 /* (Hq/Hkv) * min(8, total_tokens) query rows exceed the
                              per-KV-head row capacity (64; 32 for head_dim 256)  */
};

/* Device-detected status bits (sticky until read by pa_verify_get_device_status). */
#define PA_STATUS_QUERY_LEN 0x1u  /* a sequence has T_b > 8 (or T_b < 0)          */
#define PA_STATUS_CONTEXT   0x2u  /* past_len_b + T_b > max_context_len            */
#define PA_STATUS_BLOCK_ID  0x4u  /* a block id read is outside [0, num_blocks)    */
#define PA_STATUS_BEGINS    0x8u  /* subsequence_begins not monotone / wrong total */
#define PA_STATUS_PAST_LEN  0x10u /* past_len_b < 0                                 */
#define PA_STATUS_ROWS      0x20u /* T_b * (Hq/Hkv) above the row capacity          */
#define PA_STATUS_TIMEOUT   0x40u /* a bounded wait inside a kernel gave up         */

#define PA_MAX_QUERY_LEN 8

/* Problem dimensions. */
typedef struct {
  int32_t num_seqs;           /* B                                                   */
  int32_t total_tokens;       /* sum_b T_b = subsequence_begins[B]                    */
  int32_t num_q_heads;        /* Hq                                                  */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0, query head h uses KV head h/(Hq/Hkv) */
  int32_t head_dim;           /* D                                                   */
  int32_t page_size;          /* ps: tokens per KV page                              */
  int32_t num_blocks;         /* physical pages in each cache                        */
  int32_t max_blocks_per_seq; /* width of the block table                            */
  pa_dtype q_dtype;           /* F32, F16 or BF16                                    */
  pa_dtype out_dtype;         /* F32, F16 or BF16                                    */
} pa_dims;

/* The launch plan the partition heuristic picks (exposed for inspection). */
typedef struct {
  int32_t num_partitions;  /* P: KV partitions per (sequence, KV head), grid.x   */
  int32_t part_tokens;     /* keys per partition (multiple of the stage size)     */
  int32_t stage_keys;      /* keys staged per pipeline step                       */
  int32_t row_tiles;       /* kernel 0: n-tiles of 8 query rows per warp (1 or 2);
                              kernel 4: query-row tile N (16 or 32)               */
  int32_t kernel;          /* 0 = warp-level mma path (16-bit / u8 KV), 1 = fp32 path,
                              2 = tensor-memory (tcgen05) path, query rows on the MMA's
                              M dimension (16-bit KV with D <= 128; 8..64 query
                              rows per KV head), 4 = tensor-memory path for u8 KV,
                              keys on the MMA's M dimension (D = 128, pages of
                              16 / 32 / 64 tokens, up to 32 query rows).
                              Pages of 1, 2 or 4 tokens with 16-bit KV take
                              kernel 2 (D <= 128), gathering key rows with
                              16-byte cp.async copies instead of TMA boxes, or
                              kernel 0 (D = 256), a bulk copy per K row and
                              16-byte cp.async copies of the V rows          */
  int32_t num_sms;         /* SM count the plan was made for                       */
  int32_t ctas;            /* grid size B * Hkv * P                                */
  int32_t smem_bytes;      /* dynamic shared memory per partition CTA             */
} pa_plan;

/*
 * Storage layouts (the pages leave these open; this library fixes them):
 *  q    [total_tokens, Hq, D] in q_dtype, rows ordered by subsequence_begins.
 *  out  [total_tokens, Hq, D] in out_dtype.
 *  float / 16-bit caches: [num_blocks, Hkv, ps, D] in kv_dtype — one page of
 *       one KV head is a contiguous [ps, D] tile.
 *  u8 caches: [num_blocks, Hkv, ps*(D+4)] bytes — per page per KV head one
 *       record: ps*D code bytes, then ps fp16 scales, then ps fp16
 *       zero-points; value = (code - zero_point) * scale.  K records hold their
 *       codes slot-major (code of slot j, element d at j*D + d); V records
 *       dim-major (at d*ps + j), so that one head dimension of a page's
 *       tokens is contiguous for the P.V product.
 *  block_tables [B, max_blocks_per_seq] int32: logical page j/ps of sequence b
 *       lives in physical page block_tables[b][j/ps].
 *  past_lens [B] int32, subsequence_begins [B+1] int32 (device memory).
 *  The cache already holds the new tokens' K/V at positions past_len..past_len+T-1.
 */

/* Bytes of workspace pa_verify_forward needs for these dimensions (0 on bad
 * arguments).  Plans for the current device's SM count.  The workspace holds
 * the per-token split-KV partials and the status word; zero it once before
 * its first use (the status word must start at 0). */
size_t pa_verify_workspace_size(const pa_dims* dims, int32_t max_context_len,
                                int32_t sliding_window, pa_dtype kv_dtype);

/* The partition heuristic for an explicit SM count (host only, no CUDA call).
 * Returns PA_OK or a PA_ERR_* code for arguments pa_verify_forward would reject. */
int pa_verify_plan(const pa_dims* dims, int32_t max_context_len, int32_t sliding_window,
                   pa_dtype kv_dtype, int32_t num_sms, pa_plan* plan);

/*
 * The verify step: split-KV partition kernel (page gather once per KV head
 * for all T_b x group query rows, online softmax, fused u8 dequantisation,
 * per-token partials) followed by the per-token log-sum-exp combine.
 * max_context_len (host) must be >= past_len_b + T_b for every b; it sizes
 * the partition grid.  sliding_window = 0 means no window.  scale multiplies
 * q.k before the softmax.  Asynchronous on cuda_stream.
 */
int pa_verify_forward(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* past_lens,
                      const int32_t* subsequence_begins, int32_t max_context_len, float scale,
                      int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                      void* workspace, size_t workspace_bytes, void* cuda_stream);

/* As pa_verify_forward, and also records the page gather: for every page the
 * partition kernel fetches it adds (physical block id + 1) to
 * gather_trace[(b * Hkv + kv_head) * max_blocks_per_seq + logical_page]
 * (device int32 buffer, zeroed by the caller).  A page fetched once therefore
 * reads block_id + 1; pages never fetched stay 0. */
int pa_verify_forward_traced(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* past_lens,
                             const int32_t* subsequence_begins, int32_t max_context_len,
                             float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out,
                             const pa_dims* dims, void* workspace, size_t workspace_bytes,
                             void* cuda_stream, int32_t* gather_trace);

/* The two steps of pa_verify_forward as separate launches (same arguments),
 * so a caller can time or overlap them individually.  pa_verify_partition
 * writes the per-token partials (and the output of every sequence whose
 * context fits one partition); pa_verify_combine merges the partials of the
 * others into out.  Calling both in order equals one pa_verify_forward. */
int pa_verify_partition(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* past_lens,
                        const int32_t* subsequence_begins, int32_t max_context_len, float scale,
                        int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                        void* workspace, size_t workspace_bytes, void* cuda_stream);
int pa_verify_combine(const int32_t* past_lens, const int32_t* subsequence_begins,
                      int32_t max_context_len, int32_t sliding_window, pa_dtype kv_dtype,
                      void* out, const pa_dims* dims, void* workspace, size_t workspace_bytes,
                      void* cuda_stream);

/* pa_verify_forward for callers that cannot allocate device memory.  The
 * pages have no counterpart of this entry point; it exists for hosts that
 * cannot hand the library a workspace: for example a C-only host whose GPU
 * memory is already reserved by another runtime's pool and that has no
 * allocator to call, or a serving loop that must not call cudaMalloc once it
 * runs (cudaMalloc can synchronise the device and is not allowed while a
 * stream is being captured).
 *
 * Same arguments and results as pa_verify_forward, minus the workspace: the
 * split-KV partials live in a 16 MiB device array inside the library (held
 * by every GPU that loads the library until the process exits).  A call
 * whose partials need more than that (total_tokens x Hq x partitions x
 * (4*head_dim + 8) bytes, plus 256) returns PA_ERR_WORKSPACE; nothing is
 * allocated, on any path.  A call rejected for its arguments (any negative
 * code but PA_ERR_CUDA) enqueues nothing; the argument checks run before any
 * CUDA call.
 *
 * The first call in each device context resolves the array's device address
 * in that context (cudaGetSymbolAddress, with the device current); make that
 * first call before any stream capture, and again after a device reset,
 * which makes a new context.  Every call shares the one array: calls that
 * can overlap on the GPU (different streams without ordering between them)
 * race on it and give undefined results.  Each accepted call clears the
 * array's status word on cuda_stream before its kernels; device-detected
 * input errors still leave the affected rows zero, and their status bits are
 * not reported by this entry point. */
int pa_verify_forward_no_alloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* past_lens,
                               const int32_t* subsequence_begins, int32_t max_context_len,
                               float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out,
                               const pa_dims* dims, void* cuda_stream);

/*
 * pa_cache_update — the step just before the verify: write the new tokens'
 * K and V into their pages (the OpenVINO paged-attention op stores the new
 * tokens itself, issue 38153 "Step-by-step reproduction" step 3; u8 KV cache
 * precision, step 1).  After it, pa_verify_forward with the same past_lens /
 * subsequence_begins / block tables reads these tokens as keys
 * past_len_b .. past_len_b + T_b - 1.
 *
 *  k_new, v_new   [total_tokens, Hkv, head_dim] in src_dtype (F32, F16, BF16),
 *                 rows ordered by subsequence_begins.
 *  k_cache, v_cache  the caches, in kv_dtype, layouts as above; only the new
 *                 tokens' slots are written (for u8 also their scale and
 *                 zero-point entries).
 *  block_tables, past_lens, subsequence_begins  as for pa_verify_forward:
 *                 token i of sequence b goes to position p = past_lens[b] + i,
 *                 page block_tables[b][p / page_size], slot p % page_size.
 *  dims           num_seqs, total_tokens, num_kv_heads, head_dim (64/128/256;
 *                 u8: 128/256), page_size, num_blocks, max_blocks_per_seq are
 *                 used; num_q_heads, q_dtype and out_dtype are ignored.
 *  status         optional device uint32 (NULL: none).  A token whose slot
 *                 cannot be addressed (malformed begins, negative past_len, a
 *                 position beyond the block table, a block id outside
 *                 [0, num_blocks)) is skipped and sets PA_STATUS_BEGINS /
 *                 PA_STATUS_PAST_LEN / PA_STATUS_CONTEXT / PA_STATUS_BLOCK_ID.
 *
 * Float caches store each value rounded to nearest-even in kv_dtype.  u8
 * caches store, per token and KV head (separately for K and V), with every
 * binary32 operation rounded to nearest-even:
 *     scale = fp16((max - min) / 255)   (1.0 when that is 0 or not finite)
 *     zp    = fp16((0 - min) / scale)
 *     code  = clamp(rint(x / scale + zp), 0, 255)
 * so that (code - zp) * scale is within about half a code of x.  A token
 * whose values cluster far from zero (|min| above ~257 x (max - min))
 * overflows the fp16 zero-point and reads back non-finite.  Inputs are
 * expected finite.  The pages name the u8 precision only; this encoding is
 * the library's.  Asynchronous on cuda_stream (launched with programmatic
 * dependent launch); pointers 16-byte aligned (int32 arrays and status: 4). */
int pa_cache_update(const void* k_new, const void* v_new, pa_dtype src_dtype, void* k_cache, void* v_cache,
                    pa_dtype kv_dtype, const int32_t* block_tables, const int32_t* past_lens,
                    const int32_t* subsequence_begins, const pa_dims* dims, uint32_t* status,
                    void* cuda_stream);

/*
 * pa_verify_forward_tree — the verify step for a tree of draft tokens
 * (DDTree, OpenVINO issue 34644, both cited on the OpenVINO issue 38153
 * page): the same as pa_verify_forward except that the new tokens of a
 * sequence see each other through tree_mask instead of the causal chain.
 *
 *  tree_mask  device uint8 [total_tokens]: bit k of tree_mask[t] set = token
 *             t sees the new token k of its own sequence (key past_len_b + k);
 *             normally t's ancestors and t itself.  Past keys (j < past_len_b)
 *             are seen as in pa_verify_forward, the window counted from
 *             past_len_b + i.  A mask of bits 0..i for every token i gives
 *             exactly pa_verify_forward's result.  A row that sees no key
 *             at all is left zero.
 *
 * Other arguments, errors and the workspace as for pa_verify_forward
 * (pa_verify_workspace_size covers both entry points).  Tree masks run on the
 * library's default kernels; PA_ERR_NULL if tree_mask is NULL. */
int pa_verify_forward_tree(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                           const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                           float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                           void* workspace, size_t workspace_bytes, const uint8_t* tree_mask, void* cuda_stream);

/*
 * pa_forward_mixed — one call for a batch that mixes verify steps with
 * prefill chunks (the MIXED stage of the OpenVINO paged-attention op, issue
 * 38153 "Cause"; vLLM's decode_query_len gate on the dual-radeon-vllm page):
 * the same attention as pa_verify_forward, token i of sequence b seeing keys
 * lo_i .. past_len_b + i, but T_b may be any number of new tokens.
 *
 *  Sequences with T_b <= 8 (verify steps) run on the split-KV partition
 *  kernels and the combine, exactly as in pa_verify_forward, their partials
 *  indexed by slot b * 8 + i.  Sequences with T_b > 8 (prefill chunks) run
 *  on a prefill kernel: 128 or 256 query rows per CTA (rows / G tokens x the
 *  G heads of a KV head) streaming the block's keys once on the tensor cores
 *  (16-bit caches), or the fp32 FFMA kernel (fp32 caches); their rows are
 *  written directly.  When the chunks' blocks fill at most half the SMs
 *  (judged from total_tokens and the SM count) and max_context_len gives
 *  each piece >= 4096 keys, each block's keys are split into as many pieces
 *  (at most 16) as fit in one wave; a fourth kernel merges their partial
 *  rows.  The launches are ordered on cuda_stream.
 *
 *  Arguments as for pa_verify_forward; dims.total_tokens counts both kinds.
 *  The workspace is pa_mixed_workspace_size bytes (status word + partials
 *  for 8 token slots per sequence, + total_tokens x Hq x pieces prefill
 *  partial rows when the keys are split); its status word is shared by all
 *  the kernels.  Supported: bf16 / f16 caches with head_dim 64 or 128, pages of
 *  8 tokens or more and Hq / Hkv <= 128, or fp32 caches (any head_dim and
 *  page size); otherwise PA_ERR_UNSUPPORTED (PA_ERR_PAGE_SIZE for 16-bit
 *  caches with smaller pages).  Device errors as for pa_verify_forward,
 *  except that T_b > 8 is not one. */
size_t pa_mixed_workspace_size(const pa_dims* dims, int32_t max_context_len, int32_t sliding_window,
                               pa_dtype kv_dtype);
int pa_forward_mixed(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                     const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                     float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                     void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * pa_forward_mixed_tree — pa_forward_mixed whose verify steps are trees of
 * draft tokens: a sequence with T_b <= 8 sees its own new tokens through
 * tree_mask exactly as in pa_verify_forward_tree; prefill chunks (T_b > 8)
 * keep the causal chain and their tree_mask entries are not read.
 *
 *  tree_mask  device uint8 [total_tokens], as for pa_verify_forward_tree.
 *
 * Other arguments, errors and the workspace as for pa_forward_mixed;
 * PA_ERR_NULL if tree_mask is NULL. */
int pa_forward_mixed_tree(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          const int32_t* past_lens, const int32_t* subsequence_begins, int32_t max_context_len,
                          float scale, int32_t sliding_window, pa_dtype kv_dtype, void* out, const pa_dims* dims,
                          void* workspace, size_t workspace_bytes, const uint8_t* tree_mask, void* cuda_stream);

/* Synchronises cuda_stream, then reads and clears the workspace's status word
 * into *bits (PA_STATUS_* flags, 0 = clean). */
int pa_verify_get_device_status(void* workspace, void* cuda_stream, uint32_t* bits);

/* Static description of a PA_OK / PA_ERR_* code. */
const char* pa_verify_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* PA_VERIFY_H */
