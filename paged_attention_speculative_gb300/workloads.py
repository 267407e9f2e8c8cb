"""Seeded synthetic inputs for paged verify attention.

This module holds no attention arithmetic.  It builds, from a seed, the raw
storage a caller would hand to the library: queries, a paged K/V cache, a
block table, past lengths and subsequence begins.  Both the CUDA path (through
the binding) and the fp64 oracle consume what it builds; neither is imported
here.

Workload shapes follow the pages' workloads:
 * OpenVINO issue 38153 (Qwen-family GQA verify, u8 KV cache, T = 1..4 new
   tokens at 8k / 32k context; input convention past_lens=[L],
   subsequence_begins=[0, T], max_context_len=L+T — reproduction step 3);
 * SGLang discussion 36314 and the dual-radeon-vllm article (Gemma-4 hybrid:
   page size 64, sliding window 1024, batch 8 at 2-4k context);
 * the magik.net long-context note (128k-185k context, 9 verify queries).

Recipe (all arrays from one numpy PCG64 stream, drawn in a fixed order):
 1. a random permutation of the physical blocks; each sequence takes the next
    ceil((past_len + T) / page_size) blocks of it as its block table, the
    rest (>= 10 % extra) stay unreferenced;
 2. q ~ N(0, 1) rounded once to the query dtype;
 3. K then V ~ N(0, 1) for every stored slot, rounded once to the cache dtype,
    or for a u8 cache quantised per token per KV head by min/max:
    scale = (max - min) / 255 (1 if max == min) rounded to fp16,
    zp = clamp(rint(-min / scale), 0, 255), code = clamp(rint(x / scale + zp));
 4. poison: every slot that no query may read (unreferenced blocks, slots
    after the last new token, pages wholly before a sliding window) holds NaN
    (for u8: a NaN scale and zero-point), so a stray read shows up as NaN.
Unused block-table entries point at poisoned blocks.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import numpy as np

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "u8": 1}


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bfloat16 bit patterns, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = np.isnan(x)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 data once to the stored dtype; returns the stored bits
    (float32 for f32, uint16 patterns for f16 / bf16)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x.astype(np.float16)).view(np.uint16)
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    raise ValueError(dtype)


def storage_to_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Stored bits -> float64 values (exact)."""
    if dtype == "f32":
        return raw.astype(np.float64)
    if dtype == "f16":
        return raw.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(raw).astype(np.float64)
    raise ValueError(dtype)


def quantize_u8(x: np.ndarray):
    """Per-row (last axis) min/max u8 quantisation of the test-input recipe.

    Returns (codes uint8 [..., D], scale fp16 [...], zp fp16 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    scale = ((mx.astype(np.float64) - mn) / 255.0)
    scale = np.where(scale > 0, scale, 1.0).astype(np.float16)
    s64 = scale.astype(np.float64)
    zp = np.clip(np.rint(-mn / s64), 0, 255)
    codes = np.clip(np.rint(x / s64[..., None] + zp[..., None]), 0, 255).astype(np.uint8)
    return codes, scale, zp.astype(np.float16)


def u8_record_bytes(page_size: int, head_dim: int) -> int:
    return page_size * (head_dim + 4)


def pack_u8_records(codes: np.ndarray, scale: np.ndarray, zp: np.ndarray, dim_major: bool = False) -> np.ndarray:
    """[nb, Hkv, ps, D] codes + [nb, Hkv, ps] fp16 scale / zp -> the u8 page
    records [nb, Hkv, ps*(D+4)]: codes, then scales, then zps.  K records hold
    the codes slot-major ([ps][D]); V records (dim_major) hold them dim-major
    ([D][ps]), so one head dimension of a page's tokens is contiguous."""
    nb, hkv, ps, d = codes.shape
    rec = np.empty((nb, hkv, ps * (d + 4)), dtype=np.uint8)
    c = np.swapaxes(codes, 2, 3) if dim_major else codes
    rec[:, :, : ps * d] = np.ascontiguousarray(c).reshape(nb, hkv, ps * d)
    rec[:, :, ps * d: ps * d + 2 * ps] = np.ascontiguousarray(scale).view(np.uint8).reshape(nb, hkv, 2 * ps)
    rec[:, :, ps * d + 2 * ps:] = np.ascontiguousarray(zp).view(np.uint8).reshape(nb, hkv, 2 * ps)
    return rec


def unpack_u8_codes(rec: np.ndarray, page_size: int, head_dim: int, dim_major: bool = False) -> np.ndarray:
    """The codes of u8 page records as [nb, Hkv, ps, D] (inverse of the code
    part of pack_u8_records)."""
    nb, hkv = rec.shape[0], rec.shape[1]
    ps, d = page_size, head_dim
    c = rec.reshape(nb, hkv, ps * (d + 4))[:, :, : ps * d]
    if dim_major:
        return np.swapaxes(c.reshape(nb, hkv, d, ps), 2, 3)
    return c.reshape(nb, hkv, ps, d)


@dataclasses.dataclass
class Case:
    """One verify-step workload in raw storage form."""
    name: str
    q: np.ndarray              # [total_tokens, Hq, D] stored bits
    k_cache: np.ndarray        # [nb, Hkv, ps, D] stored bits, or u8 records [nb, Hkv, rec]
    v_cache: np.ndarray
    block_tables: np.ndarray   # [B, max_blocks_per_seq] int32
    past_lens: np.ndarray      # [B] int32
    subsequence_begins: np.ndarray  # [B + 1] int32
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_blocks: int
    q_dtype: str
    kv_dtype: str
    out_dtype: str
    scale: float
    sliding_window: int

    @property
    def num_seqs(self) -> int:
        return int(self.past_lens.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.subsequence_begins[-1])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.subsequence_begins)

    @property
    def max_context_len(self) -> int:
        t = self.query_lens
        return int((self.past_lens + t).max()) if len(t) else 0

    def kv_positions_read(self) -> np.ndarray:
        """Per sequence, the number of key positions in the union of its rows'
        key ranges (what one KV head streams once)."""
        t = self.query_lens.astype(np.int64)
        L = self.past_lens.astype(np.int64)
        n = L + t
        if self.sliding_window > 0:
            n = np.minimum(n, self.sliding_window + t - 1)
        return np.where(t > 0, n, 0)

    def kv_bytes(self) -> int:
        """Algorithmic KV-read bytes of one step: each KV head reads each key
        of the union range once (K and V; u8 adds fp16 scale + zp per key)."""
        per_key = 2 * self.head_dim * DTYPE_BYTES[self.kv_dtype] + (8 if self.kv_dtype == "u8" else 0)
        return int(self.kv_positions_read().sum()) * self.num_kv_heads * per_key

    def flops(self) -> int:
        """Algorithmic flops: 4 * D per (query row, visible key)."""
        G = self.num_q_heads // self.num_kv_heads
        tot = 0
        for b in range(self.num_seqs):
            L = int(self.past_lens[b])
            for i in range(int(self.query_lens[b])):
                p = L + i
                lo = max(0, p - self.sliding_window + 1) if self.sliding_window > 0 else 0
                tot += (p - lo + 1)
        return 4 * self.head_dim * G * self.num_kv_heads * tot


def make_case(name: str, *, seed: int, query_lens: Sequence[int], past_lens: Sequence[int],
              num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
              q_dtype: str = "bf16", kv_dtype: str = "bf16", out_dtype: str | None = None,
              sliding_window: int = 0, scale: float | None = None, extra_block_frac: float = 0.10,
              poison: bool = True, table_slack: int = 1) -> Case:
    rng = np.random.default_rng(seed)
    B = len(past_lens)
    tl = np.asarray(query_lens, dtype=np.int64)
    pl = np.asarray(past_lens, dtype=np.int64)
    assert tl.shape == (B,)
    ps, D, Hq, Hkv = page_size, head_dim, num_q_heads, num_kv_heads
    pages = [int(math.ceil((pl[b] + tl[b]) / ps)) for b in range(B)]
    max_blocks = max(pages) + table_slack if B else 1
    used = int(sum(pages))
    extra = max(2, int(math.ceil(used * extra_block_frac)))
    nb = used + extra
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.empty((B, max_blocks), dtype=np.int32)
    poisoned = list(perm[used:])
    cur = 0
    for b in range(B):
        bt[b, : pages[b]] = perm[cur: cur + pages[b]]
        cur += pages[b]
        fill = [poisoned[(b + j) % len(poisoned)] for j in range(max_blocks - pages[b])]
        bt[b, pages[b]:] = np.asarray(fill, dtype=np.int32)
    begins = np.zeros(B + 1, dtype=np.int32)
    begins[1:] = np.cumsum(tl)
    total_tokens = int(begins[-1])

    q = to_storage(rng.standard_normal((total_tokens, Hq, D), dtype=np.float32), q_dtype)

    # Which (block, slot) pairs hold readable data.
    valid = np.zeros((nb, ps), dtype=bool)
    for b in range(B):
        L, T = int(pl[b]), int(tl[b])
        n = L + T
        first_read_page = 0
        if sliding_window > 0 and poison:
            first_read_page = max(0, L - sliding_window + 1) // ps
        for lp in range(pages[b]):
            lo_slot = lp * ps
            cnt = min(ps, n - lo_slot)
            if lp < first_read_page:
                continue
            valid[bt[b, lp], :cnt] = True
    if not poison:
        valid[:] = True

    def draw_cache(dim_major):
        x = rng.standard_normal((nb, Hkv, ps, D), dtype=np.float32)
        if kv_dtype == "u8":
            codes, s, z = quantize_u8(x)
            bad = ~valid
            s[np.broadcast_to(bad[:, None, :], s.shape)] = np.float16(np.nan)
            z[np.broadcast_to(bad[:, None, :], z.shape)] = np.float16(np.nan)
            return pack_u8_records(codes, s, z, dim_major=dim_major)
        x[np.broadcast_to(~valid[:, None, :, None], x.shape)] = np.nan
        return to_storage(x, kv_dtype)

    k = draw_cache(False)
    v = draw_cache(True)  # u8 V records hold their codes dim-major
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return Case(name=name, q=q, k_cache=k, v_cache=v, block_tables=bt, past_lens=pl.astype(np.int32),
                subsequence_begins=begins, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                page_size=ps, num_blocks=nb, q_dtype=q_dtype, kv_dtype=kv_dtype,
                out_dtype=out_dtype or ("f32" if q_dtype == "f32" else q_dtype), scale=float(scale),
                sliding_window=int(sliding_window))


# ---------------------------------------------------------------------------
# The five workload families (sizes as stated with each constructor).
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Case:
    """1 sequence, past_len 512, T=3, 8 q heads / 2 KV heads, D=64, page 16, fp32."""
    return make_case("tiny", seed=seed, query_lens=[3], past_lens=[512], num_q_heads=8,
                     num_kv_heads=2, head_dim=64, page_size=16, q_dtype="f32", kv_dtype="f32")


def _ps_tag(page_size: int) -> str:
    return "" if page_size == 16 else f"_ps{page_size}"


def qwen_gqa(T: int, L: int, seed: int = 0, page_size: int = 16, **kw) -> Case:
    """Qwen-like GQA verify: batch 1, 32 q / 8 KV heads, D=128, page 16, bf16."""
    return make_case(f"qwen_gqa_T{T}_L{L}{_ps_tag(page_size)}", seed=seed, query_lens=[T], past_lens=[L],
                     num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=page_size, **kw)


def qwen_u8(T: int, L: int, seed: int = 0, **kw) -> Case:
    """Same shapes as qwen_gqa with a u8 KV cache (per-token fp16 scale / zp)."""
    kw.setdefault("q_dtype", "bf16")
    return make_case(f"qwen_u8_T{T}_L{L}", seed=seed, query_lens=[T], past_lens=[L], num_q_heads=32,
                     num_kv_heads=8, head_dim=128, page_size=16, kv_dtype="u8", **kw)


def gemma_hybrid(L: int, window: int = 0, T: int = 2, seed: int = 0, **kw) -> Case:
    """Gemma-like hybrid layer: 32 q / 16 KV heads, D=256, page 64, bf16, batch 1."""
    tag = f"swa{window}" if window else "global"
    return make_case(f"gemma_{tag}_T{T}_L{L}", seed=seed, query_lens=[T], past_lens=[L], num_q_heads=32,
                     num_kv_heads=16, head_dim=256, page_size=64, sliding_window=window, **kw)


def batched_mix_a(seed: int = 0, **kw) -> Case:
    """Batch 8, T ~ U{1..4}, past_len ~ U[2000, 4000], window 1024,
    32 q / 16 KV heads, D=256, page 64, bf16."""
    r = np.random.default_rng(1000 + seed)
    T = r.integers(1, 5, size=8)
    L = r.integers(2000, 4001, size=8)
    return make_case("mix_a", seed=seed, query_lens=T.tolist(), past_lens=L.tolist(), num_q_heads=32,
                     num_kv_heads=16, head_dim=256, page_size=64, sliding_window=1024, **kw)


def long_ctx_b(L: int, T: int = 8, seed: int = 0, page_size: int = 16, **kw) -> Case:
    """Batch 1, T=8, 64 q / 8 KV heads, D=128, page 16, bf16 (128k-185k context).
    page_size=1 is the one-token-per-page layout of the long-context stress
    case (every key its own block-table lookup)."""
    return make_case(f"long_T{T}_L{L}{_ps_tag(page_size)}", seed=seed, query_lens=[T], past_lens=[L],
                     num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=page_size, **kw)


def relayout(case: Case, page_size: int, seed: int = 0) -> Case:
    """The same logical K/V (float or 16-bit caches) in pages of `page_size`
    tokens: a fresh shuffled block table, every unreferenced slot NaN."""
    assert case.kv_dtype != "u8"
    ps0, ps = case.page_size, page_size
    rng = np.random.default_rng(seed)
    n_tok = (case.past_lens.astype(np.int64) + case.query_lens.astype(np.int64))
    pages = [int(math.ceil(int(n) / ps)) for n in n_tok]
    used = int(sum(pages))
    nb = used + max(2, used // 10)
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = max(pages) + 1
    bt = np.empty((case.num_seqs, max_blocks), dtype=np.int32)
    shape = (nb, case.num_kv_heads, ps, case.head_dim)
    k = to_storage(np.full(shape, np.nan, dtype=np.float32), case.kv_dtype)
    v = k.copy()
    cur = 0
    for b in range(case.num_seqs):
        bt[b, : pages[b]] = perm[cur: cur + pages[b]]
        spare = perm[used:]  # unreferenced (all-NaN) blocks fill the table's tail
        bt[b, pages[b]:] = spare[np.arange(max_blocks - pages[b]) % len(spare)]
        cur += pages[b]
        j = np.arange(int(n_tok[b]))
        src_blk, src_slot = case.block_tables[b][j // ps0], j % ps0
        dst_blk, dst_slot = bt[b][j // ps], j % ps
        k[dst_blk, :, dst_slot] = case.k_cache[src_blk, :, src_slot]
        v[dst_blk, :, dst_slot] = case.v_cache[src_blk, :, src_slot]
    return dataclasses.replace(case, name=f"{case.name}_as_ps{ps}", k_cache=k, v_cache=v, block_tables=bt,
                               page_size=ps, num_blocks=nb)


def new_tokens(case: Case, src_dtype: str = "bf16", seed: int = 0, specials: bool = False):
    """The new tokens' K and V for a cache-update test: [total_tokens, Hkv, D]
    ~ N(0, 1), rounded once to src_dtype (stored bits).  With specials, a few
    (token, head) rows are replaced by shapes the u8 encoding must handle: a
    constant row, an all-negative row, an all-positive row, and a row with a
    single outlier."""
    rng = np.random.default_rng(np.random.PCG64(seed + 7919))
    T = int(case.subsequence_begins[-1])
    shape = (T, case.num_kv_heads, case.head_dim)
    out = []
    for _ in range(2):
        x = rng.standard_normal(shape).astype(np.float32)
        if specials and T > 0:
            rows = [(t, h) for t in range(T) for h in range(case.num_kv_heads)]
            picks = rng.permutation(len(rows))[:4]
            kinds = ["constant", "negative", "positive", "outlier"]
            for k, i in zip(kinds, picks):
                t, h = rows[i]
                if k == "constant":
                    x[t, h] = np.float32(0.75)
                elif k == "negative":
                    x[t, h] = -2.0 - np.abs(x[t, h])
                elif k == "positive":
                    x[t, h] = 1.0 + np.abs(x[t, h])
                else:
                    x[t, h, rng.integers(case.head_dim)] = np.float32(40.0)
        out.append(to_storage(x, src_dtype))
    return out[0], out[1]
