"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: hand-derived golden
values, an independent dense brute force (materialised mask + full softmax),
a library attention routine on the T=1 case, closed forms (W=1, q=0, equal
keys, a window covering everything), the invariant that a T-token verify
equals T single-token decodes with key limits past_len+i+1 (OpenVINO issue
38153, Suggestion paragraph), block-table permutation, causal and window
perturbation, the convex-hull bound, and u8 == float on the dequantised cache;
for prefill chunks and mixed batches, the dense brute force, torch's causal
attention at past_len 0, single-token decodes beyond 32 new tokens, and the
independence of a batch's sequences.
"""
import json
import math
import os

import numpy as np
import pytest

from paged_attention_speculative_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


# ---------------------------------------------------------------------------
# Independent dense brute force (numpy).  Written from the definition with
# whole-sequence gathers and a materialised [T, n] mask; no loops over keys.
# ---------------------------------------------------------------------------

def _decode_cache(case):
    """-> float64 [nb, Hkv, ps, D] values of the stored cache."""
    ps, D = case.page_size, case.head_dim
    if case.kv_dtype != "u8":
        return (W.storage_to_f64(case.k_cache, case.kv_dtype).reshape(case.num_blocks, case.num_kv_heads, ps, D),
                W.storage_to_f64(case.v_cache, case.kv_dtype).reshape(case.num_blocks, case.num_kv_heads, ps, D))
    out = []
    for rec, dim_major in ((case.k_cache, False), (case.v_cache, True)):
        rec = rec.reshape(case.num_blocks, case.num_kv_heads, ps * (D + 4))
        codes = W.unpack_u8_codes(rec, ps, D, dim_major=dim_major).astype(np.float64)
        sc = np.ascontiguousarray(rec[:, :, ps * D: ps * D + 2 * ps]).view(np.float16).astype(np.float64)
        zp = np.ascontiguousarray(rec[:, :, ps * D + 2 * ps:]).view(np.float16).astype(np.float64)
        out.append((codes - zp[..., None]) * sc[..., None])
    return tuple(out)


def brute_force(case):
    kc, vc = _decode_cache(case)
    q = W.storage_to_f64(case.q, case.q_dtype).reshape(case.total_tokens, case.num_q_heads, case.head_dim)
    G = case.num_q_heads // case.num_kv_heads
    out = np.zeros_like(q)
    for b in range(case.num_seqs):
        T = int(case.query_lens[b])
        if T == 0:
            continue
        L = int(case.past_lens[b])
        n = L + T
        pos = np.arange(n)
        blocks = case.block_tables[b][pos // case.page_size]
        Kseq = kc[blocks, :, pos % case.page_size, :]          # [n, Hkv, D]
        Vseq = vc[blocks, :, pos % case.page_size, :]
        Kh = np.repeat(Kseq, G, axis=1).transpose(1, 0, 2)     # [Hq, n, D]
        Vh = np.repeat(Vseq, G, axis=1).transpose(1, 0, 2)
        t0 = int(case.subsequence_begins[b])
        Qb = q[t0: t0 + T].transpose(1, 0, 2)                   # [Hq, T, D]
        S = case.scale * np.einsum("htd,hnd->htn", Qb, Kh)
        i = np.arange(T)[:, None]
        j = pos[None, :]
        allowed = j <= L + i
        if case.sliding_window > 0:
            allowed &= j >= L + i - case.sliding_window + 1
        S = np.where(allowed[None], S, -np.inf)
        S = S - S.max(axis=-1, keepdims=True)
        P = np.exp(S)
        P = P / P.sum(axis=-1, keepdims=True)
        # keys no row may see carry weight exactly 0: drop them (their stored
        # values may be NaN-poisoned and 0 * NaN would leak into the sum)
        seen = allowed.any(axis=0)
        out[t0: t0 + T] = np.einsum("htn,hnd->htd", P[:, :, seen], Vh[:, seen]).transpose(1, 0, 2)
    return out


def run_oracle(oracle_mod, case, **over):
    kw = dict(num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
              page_size=case.page_size, num_blocks=case.num_blocks, scale=case.scale,
              sliding_window=case.sliding_window)
    kw.update(over)
    return oracle_mod.forward(case.q, case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype,
                              case.block_tables, case.past_lens, case.subsequence_begins, **kw)


def small_cases():
    return [
        W.make_case("tiny_f32", seed=1, query_lens=[3], past_lens=[40], num_q_heads=8, num_kv_heads=2,
                    head_dim=16, page_size=16, q_dtype="f32", kv_dtype="f32"),
        W.make_case("bf16_gqa", seed=2, query_lens=[4], past_lens=[70], num_q_heads=8, num_kv_heads=2,
                    head_dim=32, page_size=16),
        W.make_case("f16_win", seed=3, query_lens=[3], past_lens=[90], num_q_heads=4, num_kv_heads=2,
                    head_dim=16, page_size=8, q_dtype="f16", kv_dtype="f16", sliding_window=20),
        W.make_case("u8", seed=4, query_lens=[3], past_lens=[50], num_q_heads=4, num_kv_heads=1,
                    head_dim=32, page_size=16, kv_dtype="u8"),
        W.make_case("batch_mixed_T", seed=5, query_lens=[1, 0, 4, 2], past_lens=[9, 30, 33, 0],
                    num_q_heads=6, num_kv_heads=3, head_dim=16, page_size=4, sliding_window=7),
        W.make_case("u8_win_batch", seed=6, query_lens=[2, 3], past_lens=[64, 17], num_q_heads=4,
                    num_kv_heads=2, head_dim=16, page_size=8, kv_dtype="u8", q_dtype="f16", sliding_window=10),
    ]


@pytest.mark.parametrize("idx", range(6))
def test_oracle_matches_dense_brute_force(oracle_mod, idx):
    case = small_cases()[idx]
    got = run_oracle(oracle_mod, case)
    want = brute_force(case)
    assert np.isfinite(got).all(), "oracle read a poisoned slot"
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Hand-derived golden values.
# ---------------------------------------------------------------------------

def _golden_case(c, kv_dtype="f32", codes=None):
    Hq, Hkv, D, ps = c["num_q_heads"], c["num_kv_heads"], c["head_dim"], c["page_size"]
    nb = c["num_blocks"]
    bt = np.array(c["block_tables"], dtype=np.int32)
    if "k_positions_per_head" in c:
        kpos = np.array(c["k_positions_per_head"], dtype=np.float32)   # [Hkv, n, D]
        vpos = np.array(c["v_positions_per_head"], dtype=np.float32)
    else:
        kpos = np.repeat(np.array(c["k_positions"], dtype=np.float32)[None], Hkv, axis=0)
        vpos = np.repeat(np.array(c["v_positions"], dtype=np.float32)[None], Hkv, axis=0)
    n = kpos.shape[1]
    kc = np.zeros((nb, Hkv, ps, D), dtype=np.float32)
    vc = np.zeros((nb, Hkv, ps, D), dtype=np.float32)
    for j in range(n):
        blk = bt[0][j // ps]
        kc[blk, :, j % ps] = kpos[:, j]
        vc[blk, :, j % ps] = vpos[:, j]
    q = np.array(c["q"], dtype=np.float32)
    return q, kc, vc, bt


def test_golden_hand_worked(oracle_mod):
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        q, kc, vc, bt = _golden_case(c)
        got = oracle_mod.forward(q, "f32", kc, vc, "f32", bt, c["past_lens"], c["subsequence_begins"],
                                 num_q_heads=c["num_q_heads"], num_kv_heads=c["num_kv_heads"],
                                 head_dim=c["head_dim"], page_size=c["page_size"],
                                 num_blocks=c["num_blocks"], scale=math.log(2.0),
                                 sliding_window=c["sliding_window"])
        np.testing.assert_allclose(got, np.array(c["expected"]), rtol=0, atol=1e-12, err_msg=c["name"])


def test_golden_u8_records(oracle_mod):
    g = json.load(open(GOLDEN))
    c = g["cases"][0]
    u = g["u8_case"]
    ps, D, nb = c["page_size"], c["head_dim"], c["num_blocks"]
    bt = np.array(c["block_tables"], dtype=np.int32)
    codes_k = np.zeros((nb, 1, ps, D), np.uint8)
    codes_v = np.zeros((nb, 1, ps, D), np.uint8)
    for j, (ck, cv) in enumerate(zip(u["k_codes_positions"], u["v_codes_positions"])):
        blk = bt[0][j // ps]
        codes_k[blk, 0, j % ps] = ck
        codes_v[blk, 0, j % ps] = cv
    sc = np.full((nb, 1, ps), u["scale_fp16"], np.float16)
    zp = np.full((nb, 1, ps), u["zp_fp16"], np.float16)
    kr = W.pack_u8_records(codes_k, sc, zp)
    vr = W.pack_u8_records(codes_v, sc, zp, dim_major=True)
    q = np.array(c["q"], dtype=np.float32)
    got = oracle_mod.forward(q, "f32", kr, vr, "u8", bt, c["past_lens"], c["subsequence_begins"],
                             num_q_heads=1, num_kv_heads=1, head_dim=D, page_size=ps, num_blocks=nb,
                             scale=math.log(2.0), sliding_window=0)
    np.testing.assert_allclose(got, np.array(u["expected"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Library routine on the T = 1 case (plain attention over all L+1 keys).
# ---------------------------------------------------------------------------

def test_t1_matches_torch_sdpa(oracle_mod):
    torch = pytest.importorskip("torch")
    case = W.make_case("t1", seed=11, query_lens=[1], past_lens=[77], num_q_heads=8, num_kv_heads=2,
                       head_dim=32, page_size=16)
    got = run_oracle(oracle_mod, case)
    kc, vc = _decode_cache(case)
    n = 78
    pos = np.arange(n)
    blocks = case.block_tables[0][pos // 16]
    K = torch.from_numpy(kc[blocks, :, pos % 16, :].transpose(1, 0, 2).copy())   # [Hkv, n, D]
    V = torch.from_numpy(vc[blocks, :, pos % 16, :].transpose(1, 0, 2).copy())
    K = K.repeat_interleave(4, dim=0)
    V = V.repeat_interleave(4, dim=0)
    q = torch.from_numpy(W.storage_to_f64(case.q, "bf16").reshape(1, 8, 32).transpose(1, 0, 2).copy())
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], K[None], V[None], scale=case.scale)[0]
    np.testing.assert_allclose(got[0], ref.numpy().transpose(1, 0, 2)[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# The equivalence the pages state: T-token verify == T single-token decodes.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("window", [0, 13])
def test_t_tokens_equal_t_single_token_decodes(oracle_mod, window):
    case = W.make_case("eq", seed=21, query_lens=[5], past_lens=[41], num_q_heads=6, num_kv_heads=2,
                       head_dim=16, page_size=8, sliding_window=window)
    multi = run_oracle(oracle_mod, case)
    for i in range(5):
        # token i alone, as a single-token decode with past_len L+i
        single = oracle_mod.forward(case.q[i: i + 1], case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype,
                                    case.block_tables, [41 + i], [0, 1], num_q_heads=6, num_kv_heads=2,
                                    head_dim=16, page_size=8, num_blocks=case.num_blocks, scale=case.scale,
                                    sliding_window=window)
        assert np.array_equal(multi[i], single[0])


# ---------------------------------------------------------------------------
# Closed forms.
# ---------------------------------------------------------------------------

def test_window_one_returns_own_value(oracle_mod):
    case = W.make_case("w1", seed=31, query_lens=[4], past_lens=[20], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8, sliding_window=1, poison=False)
    got = run_oracle(oracle_mod, case)
    _, vc = _decode_cache(case)
    for i in range(4):
        p = 20 + i
        blk = case.block_tables[0][p // 8]
        for h in range(4):
            assert np.array_equal(got[i, h], vc[blk, h // 2, p % 8])


def test_zero_query_gives_mean_of_visible_values(oracle_mod):
    case = W.make_case("q0", seed=32, query_lens=[3], past_lens=[25], num_q_heads=2, num_kv_heads=1,
                       head_dim=8, page_size=4, sliding_window=9)
    case.q[:] = 0
    got = run_oracle(oracle_mod, case)
    _, vc = _decode_cache(case)
    for i in range(3):
        p = 25 + i
        js = np.arange(p - 8, p + 1)
        vals = vc[case.block_tables[0][js // 4], 0, js % 4]
        np.testing.assert_allclose(got[i, 0], vals.mean(axis=0), rtol=0, atol=1e-13)


def test_equal_keys_give_mean(oracle_mod):
    case = W.make_case("eqk", seed=33, query_lens=[2], past_lens=[10], num_q_heads=2, num_kv_heads=1,
                       head_dim=8, page_size=4, q_dtype="f32", kv_dtype="f32", poison=False)
    kc = case.k_cache.reshape(case.num_blocks, 1, 4, 8)
    kc[:] = kc[0, 0, 0]
    got = run_oracle(oracle_mod, case)
    _, vc = _decode_cache(case)
    for i in range(2):
        js = np.arange(0, 11 + i)
        vals = vc[case.block_tables[0][js // 4], 0, js % 4]
        np.testing.assert_allclose(got[i, 0], vals.mean(axis=0), rtol=0, atol=1e-12)


def test_window_covering_everything_equals_no_window(oracle_mod):
    case = W.make_case("wbig", seed=34, query_lens=[3], past_lens=[30], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8)
    a = run_oracle(oracle_mod, case)
    b = run_oracle(oracle_mod, case, sliding_window=33)
    c = run_oracle(oracle_mod, case, sliding_window=10_000)
    assert np.array_equal(a, b) and np.array_equal(a, c)


# ---------------------------------------------------------------------------
# Invariants.
# ---------------------------------------------------------------------------

def test_block_table_permutation_moves_pages(oracle_mod):
    case = W.make_case("perm", seed=41, query_lens=[3], past_lens=[45], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8)
    a = run_oracle(oracle_mod, case)
    rng = np.random.default_rng(7)
    perm = rng.permutation(case.num_blocks)       # new physical id of each old block
    inv = np.argsort(perm)
    k2 = case.k_cache.reshape(case.num_blocks, -1)[inv].copy()
    v2 = case.v_cache.reshape(case.num_blocks, -1)[inv].copy()
    bt2 = perm[case.block_tables].astype(np.int32)
    b = oracle_mod.forward(case.q, case.q_dtype, k2, v2, case.kv_dtype, bt2, case.past_lens,
                           case.subsequence_begins, num_q_heads=4, num_kv_heads=2, head_dim=16, page_size=8,
                           num_blocks=case.num_blocks, scale=case.scale)
    assert np.array_equal(a, b)


def test_future_and_out_of_window_keys_do_not_matter(oracle_mod):
    L, T, Wn, ps = 30, 4, 6, 8
    case = W.make_case("pert", seed=42, query_lens=[T], past_lens=[L], num_q_heads=2, num_kv_heads=1,
                       head_dim=8, page_size=ps, q_dtype="f32", kv_dtype="f32", sliding_window=Wn)
    a = run_oracle(oracle_mod, case)
    kc = case.k_cache.reshape(case.num_blocks, 1, ps, 8)
    vc = case.v_cache.reshape(case.num_blocks, 1, ps, 8)
    # change the last new token's key/value: only token T-1 may move
    p_last = L + T - 1
    blk = case.block_tables[0][p_last // ps]
    kc[blk, 0, p_last % ps] += 3.0
    vc[blk, 0, p_last % ps] -= 5.0
    b = run_oracle(oracle_mod, case)
    assert np.array_equal(a[: T - 1], b[: T - 1])
    assert not np.array_equal(a[T - 1], b[T - 1])
    # change the key just before token 2's window: tokens >= 2 stay, token 1 moves
    j = L + 2 - Wn
    blk = case.block_tables[0][j // ps]
    vc[blk, 0, j % ps] += 7.0
    c = run_oracle(oracle_mod, case)
    assert np.array_equal(b[2:], c[2:])
    assert not np.array_equal(b[1], c[1])


def test_output_inside_value_hull(oracle_mod):
    case = small_cases()[1]
    got = run_oracle(oracle_mod, case)
    _, vc = _decode_cache(case)
    L = int(case.past_lens[0])
    for i in range(int(case.query_lens[0])):
        js = np.arange(0, L + i + 1)
        for h in range(case.num_q_heads):
            vals = vc[case.block_tables[0][js // 16], h // 4, js % 16]
            assert (got[i, h] >= vals.min(axis=0) - 1e-12).all()
            assert (got[i, h] <= vals.max(axis=0) + 1e-12).all()


def test_u8_equals_float_on_dequantised_cache(oracle_mod):
    case = W.make_case("u8deq", seed=51, query_lens=[3], past_lens=[37], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8, kv_dtype="u8", q_dtype="f32")
    a = run_oracle(oracle_mod, case)
    kc, vc = _decode_cache(case)
    b = oracle_mod.forward(case.q, "f32", kc.astype(np.float32), vc.astype(np.float32), "f32",
                           case.block_tables, case.past_lens, case.subsequence_begins, num_q_heads=4,
                           num_kv_heads=2, head_dim=16, page_size=8, num_blocks=case.num_blocks,
                           scale=case.scale)
    finite = np.isfinite(a)
    assert finite.all()
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-6)


# ---------------------------------------------------------------------------
# Stored-value decoding over every 16-bit pattern (single visible key: out = V).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_every_16bit_pattern_decodes_exactly(oracle_mod, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = W.storage_to_f64(bits, dtype)
    keep = np.isfinite(vals)
    bits, vals = bits[keep], vals[keep]
    n = bits.shape[0]
    # n sequences, each L=0, T=1, its own page (page_size 1, D=1); V holds one pattern.
    bt = np.arange(n, dtype=np.int32)[:, None]
    q = np.zeros((n, 1, 1), dtype=np.uint16)
    k = np.zeros((n, 1, 1, 1), dtype=np.uint16)
    v = bits.reshape(n, 1, 1, 1)
    got = oracle_mod.forward(q, dtype, k, v, dtype, bt, np.zeros(n, np.int32), np.arange(n + 1, dtype=np.int32),
                             num_q_heads=1, num_kv_heads=1, head_dim=1, page_size=1, num_blocks=n, scale=1.0)
    assert np.array_equal(got.reshape(n), vals)


# ---------------------------------------------------------------------------
# Pages touched: brute force over every row's key range.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("idx", range(6))
def test_pages_touched_brute_force(oracle_mod, idx):
    case = small_cases()[idx]
    got = oracle_mod.pages_touched(case.block_tables, case.past_lens, case.subsequence_begins,
                                   page_size=case.page_size, sliding_window=case.sliding_window)
    want = np.zeros_like(case.block_tables)
    for b in range(case.num_seqs):
        L = int(case.past_lens[b])
        for i in range(int(case.query_lens[b])):
            p = L + i
            lo = max(0, p - case.sliding_window + 1) if case.sliding_window > 0 else 0
            for j in range(lo, p + 1):
                want[b, j // case.page_size] = case.block_tables[b, j // case.page_size] + 1
    assert np.array_equal(got, want)


def test_bad_block_id_is_reported(oracle_mod):
    case = small_cases()[1]
    case.block_tables[0, 1] = case.num_blocks + 5
    with pytest.raises(ValueError):
        run_oracle(oracle_mod, case)


def test_workload_families_have_stated_shapes():
    c = W.tiny()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.page_size, c.total_tokens) == (8, 2, 64, 16, 3)
    assert c.q_dtype == "f32" and int(c.past_lens[0]) == 512
    a = W.batched_mix_a()
    assert a.num_seqs == 8 and a.sliding_window == 1024
    assert ((a.query_lens >= 1) & (a.query_lens <= 4)).all()
    assert ((a.past_lens >= 2000) & (a.past_lens <= 4000)).all()


# ---------------------------------------------------------------------------
# Cache update (the step before the verify: the new tokens' K/V written into
# their pages, with per-token u8 quantisation for u8 caches).
# ---------------------------------------------------------------------------
def _cu_layout(D=4, ps=4, num_blocks=1):
    return dict(num_kv_heads=1, head_dim=D, page_size=ps, num_blocks=num_blocks)


def _cu_one_token(oracle, x, kv_dtype, D=4, ps=4):
    """Write one f32 token x (K = V = x) at slot 1 of the only page."""
    kn = np.asarray(x, dtype=np.float32).reshape(1, 1, D)
    if kv_dtype == "u8":
        cache = np.zeros((1, 1, ps * (D + 4)), dtype=np.uint8)
    elif kv_dtype == "f32":
        cache = np.zeros((1, 1, ps, D), dtype=np.float32)
    else:
        cache = np.zeros((1, 1, ps, D), dtype=np.uint16)
    kc, vc = oracle.cache_update(kn, kn, "f32", cache, cache, kv_dtype, [[0]], [1], [0, 1], **_cu_layout(D, ps))
    if kv_dtype == "u8":
        # the V record holds the same codes dim-major, and the same scales and zero-points
        kcodes = W.unpack_u8_codes(kc.reshape(1, 1, -1), ps, D)
        vcodes = W.unpack_u8_codes(vc.reshape(1, 1, -1), ps, D, dim_major=True)
        assert np.array_equal(kcodes, vcodes)
        assert np.array_equal(kc.reshape(-1)[ps * D:], vc.reshape(-1)[ps * D:])
    else:
        assert np.array_equal(kc, vc)
    return kc


def _u8_slot(rec, slot, D, ps):
    rec = rec.reshape(-1)
    codes = rec[slot * D:(slot + 1) * D]
    scale = rec[ps * D + 2 * slot: ps * D + 2 * slot + 2].view(np.uint16)[0]
    zp = rec[ps * D + 2 * ps + 2 * slot: ps * D + 2 * ps + 2 * slot + 2].view(np.uint16)[0]
    return codes, int(scale), int(zp)


def test_cache_update_u8_hand_worked(oracle_mod):
    g = json.load(open(os.path.join(os.path.dirname(GOLDEN), "cache_update.json")))
    for case in g["u8"]:
        rec = _cu_one_token(oracle_mod, case["x"], "u8")
        codes, s, z = _u8_slot(rec, 1, 4, 4)
        assert s == case["scale_bits"] and z == case["zp_bits"], case["name"]
        assert codes.tolist() == case["codes"], case["name"]
        # the other slots are untouched
        assert not rec.reshape(-1)[:4].any() and not rec.reshape(-1)[8:16].any()


def test_cache_update_float_rounding_hand_worked(oracle_mod):
    g = json.load(open(os.path.join(os.path.dirname(GOLDEN), "cache_update.json")))
    for kv in ("f16", "bf16"):
        for case in g[kv]:
            x = np.array([case["x_f32_bits"]] * 4, dtype=np.uint32).view(np.float32)
            c = _cu_one_token(oracle_mod, x, kv)
            assert c[0, 0, 1].tolist() == [case["bits"]] * 4, (kv, case)
    x = np.array([0.1, -2.5, 3e-30, 7.0], dtype=np.float32)
    assert np.array_equal(_cu_one_token(oracle_mod, x, "f32")[0, 0, 1], x)  # f32 caches store the value itself


def test_cache_update_u8_properties(oracle_mod):
    """Round trip within half a code (plus the fp16 zero-point's rounding),
    order preserved, and the extremes at codes 0 and 255."""
    rng = np.random.default_rng(11)
    D, ps = 128, 16
    for trial in range(200):
        # offsets relative to the spread, so -min / scale stays inside fp16
        sigma = rng.choice([0.01, 1.0, 30.0])
        shift = rng.choice([0.0, -5.0, 5.0, 40.0]) * sigma
        x = (rng.standard_normal(D) * sigma + shift).astype(np.float32)
        rec = _cu_one_token(oracle_mod, x, "u8", D=D, ps=ps)
        codes, s, z = _u8_slot(rec, 1, D, ps)
        sf = float(np.array([s], dtype=np.uint16).view(np.float16)[0])
        zf = float(np.array([z], dtype=np.uint16).view(np.float16)[0])
        back = (codes.astype(np.float64) - zf) * sf
        zp_ulp = float(np.spacing(np.float16(abs(zf)))) if zf != 0 else 0.0
        bound = (0.5 + zp_ulp / 2 + 1e-3) * sf
        assert np.max(np.abs(back - x)) <= bound, trial
        order = np.argsort(x, kind="stable")
        assert np.all(np.diff(codes[order].astype(int)) >= 0), trial
        # the extremes sit at codes 0 and 255, give or take the zero-point's
        # fp16 rounding (at most half its spacing in code units)
        slack = int(zp_ulp / 2 + 0.5)
        assert codes[np.argmin(x)] <= slack and codes[np.argmax(x)] >= 255 - slack, trial


def test_cache_update_places_tokens_where_the_verify_reads_them(oracle_mod):
    """f32 cache full of NaN; the update writes T tokens per sequence; the
    (pinned) attention definition over the updated cache must equal a dense
    numpy attention over the same keys -- any misplaced token shows as NaN or
    a wrong value."""
    rng = np.random.default_rng(12)
    Hq, Hkv, D, ps = 4, 2, 8, 4
    past = [5, 0, 9]
    Ts = [3, 2, 4]
    begins = np.concatenate([[0], np.cumsum(Ts)]).astype(np.int32)
    mb = 4
    nb = 1 + len(past) * mb
    perm = rng.permutation(nb - 1) + 1
    bt = perm[: len(past) * mb].reshape(len(past), mb).astype(np.int32)
    k_dense = [rng.standard_normal((past[b] + Ts[b], Hkv, D)).astype(np.float32) for b in range(len(past))]
    v_dense = [rng.standard_normal((past[b] + Ts[b], Hkv, D)).astype(np.float32) for b in range(len(past))]
    kc = np.full((nb, Hkv, ps, D), np.nan, dtype=np.float32)
    vc = kc.copy()
    for b in range(len(past)):  # the past keys, placed by hand
        for j in range(past[b]):
            kc[bt[b, j // ps], :, j % ps] = k_dense[b][j]
            vc[bt[b, j // ps], :, j % ps] = v_dense[b][j]
    k_new = np.concatenate([k_dense[b][past[b]:] for b in range(len(past))])
    v_new = np.concatenate([v_dense[b][past[b]:] for b in range(len(past))])
    kc2, vc2 = oracle_mod.cache_update(k_new, v_new, "f32", kc, vc, "f32", bt, past, begins, num_kv_heads=Hkv,
                                   head_dim=D, page_size=ps, num_blocks=nb)
    q = rng.standard_normal((int(begins[-1]), Hq, D)).astype(np.float32)
    got = oracle_mod.forward(q, "f32", kc2, vc2, "f32", bt, past, begins, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, page_size=ps, num_blocks=nb, scale=0.35)
    G = Hq // Hkv
    for b in range(len(past)):
        for i in range(Ts[b]):
            t = begins[b] + i
            for h in range(Hq):
                keys = k_dense[b][: past[b] + i + 1, h // G].astype(np.float64)
                vals = v_dense[b][: past[b] + i + 1, h // G].astype(np.float64)
                s = 0.35 * keys @ q[t, h].astype(np.float64)
                w = np.exp(s - s.max())
                assert np.allclose(got[t, h], w @ vals / w.sum(), rtol=0, atol=1e-12)
    # nothing outside the new tokens' slots changed
    touched = np.zeros(kc.shape[:3], dtype=bool)
    for b in range(len(past)):
        for i in range(Ts[b]):
            j = past[b] + i
            touched[bt[b, j // ps], :, j % ps] = True
    assert np.array_equal(np.isnan(kc2[~touched]), np.isnan(kc[~touched]))
    assert np.array_equal(kc2[~touched & ~np.isnan(kc).any(-1)], kc[~touched & ~np.isnan(kc).any(-1)])


def test_cache_update_rejects_inconsistent_inputs(oracle_mod):
    kn = np.zeros((1, 1, 4), dtype=np.float32)
    cache = np.zeros((2, 1, 4, 4), dtype=np.float32)
    with pytest.raises(ValueError):  # block id out of range
        oracle_mod.cache_update(kn, kn, "f32", cache, cache, "f32", [[5]], [0], [0, 1], num_kv_heads=1, head_dim=4,
                            page_size=4, num_blocks=2)
    with pytest.raises(ValueError):  # position beyond the block table
        oracle_mod.cache_update(kn, kn, "f32", cache, cache, "f32", [[0]], [4], [0, 1], num_kv_heads=1, head_dim=4,
                            page_size=4, num_blocks=2)


def test_cache_update_u8_zero_point_overflow_is_visible(oracle_mod):
    """A token clustered far from zero (|min| above ~257 x its range) needs a
    zero-point beyond fp16: it rounds to -inf and the slot reads back
    non-finite instead of silently wrong."""
    x = np.float32(40.0) + np.linspace(-0.01, 0.01, 8, dtype=np.float32)
    rec = _cu_one_token(oracle_mod, x, "u8", D=8, ps=4)
    codes, s, z = _u8_slot(rec, 1, 8, 4)
    assert z == 0xFC00 and not codes.any()
    sf = float(np.array([s], dtype=np.uint16).view(np.float16)[0])
    assert not np.isfinite((codes.astype(np.float64) - (-np.inf)) * sf).any()


# ---------------------------------------------------------------------------
# Tree-mask verify: the draft tokens form a tree; a token sees the past keys
# and the new tokens its mask names (itself and its ancestors).
# ---------------------------------------------------------------------------
def _chain_mask(case):
    m = np.zeros(case.total_tokens, dtype=np.uint8)
    for b in range(case.num_seqs):
        t0 = int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            m[t0 + i] = (2 << i) - 1
    return m


def _random_tree_masks(case, rng):
    """A random tree per sequence: node i's parent is a random earlier node
    (node 0 hangs off the past); the mask of i is i plus its ancestors."""
    m = np.zeros(case.total_tokens, dtype=np.uint8)
    for b in range(case.num_seqs):
        t0 = int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            parent = -1 if i == 0 else int(rng.integers(-1, i))
            m[t0 + i] = (1 << i) | (m[t0 + parent] if parent >= 0 else 0)
    return m


def test_tree_chain_mask_is_the_causal_definition(oracle_mod):
    for case in small_cases():
        want = run_oracle(oracle_mod, case)
        got = run_oracle(oracle_mod, case, tree_mask=_chain_mask(case))
        assert np.array_equal(got, want), case.name


def test_tree_mask_against_dense_brute_force(oracle_mod):
    rng = np.random.default_rng(21)
    for case in small_cases():
        m = _random_tree_masks(case, rng)
        got = run_oracle(oracle_mod, case, tree_mask=m)
        kc, vc = _decode_cache(case)
        q = W.storage_to_f64(case.q, case.q_dtype).reshape(case.total_tokens, case.num_q_heads, case.head_dim)
        G = case.num_q_heads // case.num_kv_heads
        for b in range(case.num_seqs):
            L, t0, T = int(case.past_lens[b]), int(case.subsequence_begins[b]), int(case.query_lens[b])
            for i in range(T):
                p = L + i
                lo = max(0, p - case.sliding_window + 1) if case.sliding_window > 0 else 0
                keys = [j for j in range(lo, L + T) if j < L or (m[t0 + i] >> (j - L)) & 1]
                blk = case.block_tables[b][np.array(keys) // case.page_size]
                slot = np.array(keys) % case.page_size
                for h in range(case.num_q_heads):
                    K = kc[blk, h // G, slot]
                    V = vc[blk, h // G, slot]
                    s = case.scale * (K @ q[t0 + i, h])
                    w = np.exp(s - s.max())
                    assert np.allclose(got[t0 + i, h], w @ V / w.sum(), rtol=0, atol=1e-12), case.name


def test_tree_node_equals_a_decode_over_its_path(oracle_mod):
    """The tree semantics: node i's output is a single-token decode whose
    cache holds the past followed by i's ancestors (in order) and i itself."""
    rng = np.random.default_rng(22)
    case = W.make_case("tree", seed=23, query_lens=[7], past_lens=[37], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8, q_dtype="f32", kv_dtype="f32")
    m = _random_tree_masks(case, rng)
    got = run_oracle(oracle_mod, case, tree_mask=m)
    kc, vc = _decode_cache(case)
    L, ps, Hkv, D = 37, 8, 2, 16
    for i in range(7):
        path = [k for k in range(7) if (m[i] >> k) & 1]
        n = L + len(path)
        nb = (n + ps - 1) // ps
        k_lin = np.full((nb, Hkv, ps, D), np.nan, dtype=np.float32)
        v_lin = k_lin.copy()
        for j in range(n):
            src = j if j < L else L + path[j - L]
            blk, slot = case.block_tables[0][src // ps], src % ps
            k_lin[j // ps, :, j % ps] = kc[blk, :, slot]
            v_lin[j // ps, :, j % ps] = vc[blk, :, slot]
        one = oracle_mod.forward(case.q[i:i + 1], "f32", k_lin, v_lin, "f32", [list(range(nb))], [n - 1], [0, 1],
                                 num_q_heads=4, num_kv_heads=Hkv, head_dim=D, page_size=ps, num_blocks=nb,
                                 scale=case.scale)
        assert np.array_equal(got[i], one[0]), i


def test_tree_mask_with_no_visible_key_gives_zero(oracle_mod):
    case = W.make_case("tree_empty", seed=24, query_lens=[2], past_lens=[0], num_q_heads=2, num_kv_heads=1,
                       head_dim=8, page_size=8, q_dtype="f32", kv_dtype="f32")
    got = run_oracle(oracle_mod, case, tree_mask=np.array([0, 3], dtype=np.uint8))
    assert not got[0].any() and np.isfinite(got[1]).all() and got[1].any()


def test_page_size_does_not_change_the_result(oracle_mod):
    """The same logical K/V laid out in 1-token pages (every token its own
    block, in shuffled order) and in 16-token pages gives bitwise the same
    output: the page size only changes where a key is stored."""
    big = W.make_case("ps16", seed=31, query_lens=[3, 2], past_lens=[45, 70], num_q_heads=8, num_kv_heads=2,
                      head_dim=16, page_size=16, q_dtype="f32", kv_dtype="f32")
    kc, vc = _decode_cache(big)  # [nb, Hkv, ps, D] dequantised (exact f32 here)
    rng = np.random.default_rng(32)
    n_tok = [int(big.past_lens[b]) + int(big.query_lens[b]) for b in range(big.num_seqs)]
    total = sum(n_tok)
    perm = rng.permutation(total) + 1
    k1 = np.full((total + 1, big.num_kv_heads, 1, big.head_dim), np.nan, dtype=np.float32)
    v1 = k1.copy()
    bt1 = np.zeros((big.num_seqs, max(n_tok)), dtype=np.int32)
    cur = 0
    for b in range(big.num_seqs):
        for j in range(n_tok[b]):
            blk16, slot = big.block_tables[b][j // 16], j % 16
            bt1[b, j] = perm[cur]
            k1[perm[cur], :, 0] = kc[blk16, :, slot]
            v1[perm[cur], :, 0] = vc[blk16, :, slot]
            cur += 1
    want = run_oracle(oracle_mod, big)
    got = oracle_mod.forward(big.q, big.q_dtype, k1, v1, "f32", bt1, big.past_lens, big.subsequence_begins,
                             num_q_heads=big.num_q_heads, num_kv_heads=big.num_kv_heads, head_dim=big.head_dim,
                             page_size=1, num_blocks=total + 1, scale=big.scale)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# Mixed batches: prefill chunks (many new tokens) beside verify steps.  The
# causal rule is the same for any number of new tokens: token i of sequence b
# sees keys lo_i .. past_len_b + i.
# ---------------------------------------------------------------------------

def prefill_cases():
    return [
        W.make_case("prefill_no_past", seed=61, query_lens=[40], past_lens=[0], num_q_heads=4, num_kv_heads=2,
                    head_dim=16, page_size=8, q_dtype="f32", kv_dtype="f32"),
        W.make_case("prefill_on_past", seed=62, query_lens=[70], past_lens=[25], num_q_heads=8, num_kv_heads=2,
                    head_dim=32, page_size=16),
        W.make_case("prefill_window", seed=63, query_lens=[45], past_lens=[30], num_q_heads=4, num_kv_heads=1,
                    head_dim=16, page_size=8, q_dtype="f16", kv_dtype="f16", sliding_window=19),
        W.make_case("mixed_batch", seed=64, query_lens=[1, 3, 45, 0, 33, 8, 9], past_lens=[50, 7, 12, 3, 0, 40, 21],
                    num_q_heads=6, num_kv_heads=3, head_dim=16, page_size=4),
        W.make_case("mixed_u8", seed=65, query_lens=[2, 37], past_lens=[64, 17], num_q_heads=4, num_kv_heads=2,
                    head_dim=16, page_size=8, kv_dtype="u8", q_dtype="f16"),
    ]


@pytest.mark.parametrize("idx", range(5))
def test_prefill_and_mixed_batches_match_dense_brute_force(oracle_mod, idx):
    case = prefill_cases()[idx]
    got = run_oracle(oracle_mod, case)
    want = brute_force(case)
    assert np.isfinite(got).all(), "oracle read a poisoned slot"
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [0, 9])
def test_long_t_equals_single_token_decodes(oracle_mod, window):
    """Beyond 32 new tokens (past any bit-mask width): token i of a 45-token
    chunk equals a single-token decode with past_len L + i, bit for bit."""
    T, L = 45, 20
    case = W.make_case("eq_long", seed=66, query_lens=[T], past_lens=[L], num_q_heads=4, num_kv_heads=2,
                       head_dim=16, page_size=8, sliding_window=window)
    multi = run_oracle(oracle_mod, case)
    for i in (0, 1, 30, 31, 32, 33, 44):
        single = oracle_mod.forward(case.q[i: i + 1], case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype,
                                    case.block_tables, [L + i], [0, 1], num_q_heads=4, num_kv_heads=2,
                                    head_dim=16, page_size=8, num_blocks=case.num_blocks, scale=case.scale,
                                    sliding_window=window)
        assert np.array_equal(multi[i], single[0])


def test_prefill_without_past_matches_torch_causal_sdpa(oracle_mod):
    """past_len 0: the chunk is plain causal self-attention (library routine)."""
    torch = pytest.importorskip("torch")
    T, Hq, Hkv, D, ps = 50, 8, 2, 32, 16
    case = W.make_case("causal", seed=67, query_lens=[T], past_lens=[0], num_q_heads=Hq, num_kv_heads=Hkv,
                       head_dim=D, page_size=ps)
    got = run_oracle(oracle_mod, case)
    kc, vc = _decode_cache(case)
    pos = np.arange(T)
    blocks = case.block_tables[0][pos // ps]
    K = torch.from_numpy(kc[blocks, :, pos % ps, :].transpose(1, 0, 2).copy()).repeat_interleave(Hq // Hkv, dim=0)
    V = torch.from_numpy(vc[blocks, :, pos % ps, :].transpose(1, 0, 2).copy()).repeat_interleave(Hq // Hkv, dim=0)
    q = torch.from_numpy(W.storage_to_f64(case.q, "bf16").reshape(T, Hq, D).transpose(1, 0, 2).copy())
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], K[None], V[None], is_causal=True,
                                                           scale=case.scale)[0]
    np.testing.assert_allclose(got, ref.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_mixed_batch_is_each_sequence_alone(oracle_mod):
    """Sequences of a mixed batch do not interact: each one's rows equal a
    call with that sequence alone (bit for bit)."""
    case = prefill_cases()[3]
    got = run_oracle(oracle_mod, case)
    for b in range(case.num_seqs):
        t0, t1 = int(case.subsequence_begins[b]), int(case.subsequence_begins[b + 1])
        if t1 == t0:
            continue
        alone = oracle_mod.forward(case.q[t0:t1], case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype,
                                   case.block_tables[b: b + 1], case.past_lens[b: b + 1], [0, t1 - t0],
                                   num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                                   head_dim=case.head_dim, page_size=case.page_size, num_blocks=case.num_blocks,
                                   scale=case.scale)
        assert np.array_equal(got[t0:t1], alone)


@pytest.mark.parametrize("ps", [1, 2, 4, 32])
def test_relayout_keeps_the_logical_cache(oracle_mod, ps):
    """workloads.relayout (used by the GPU page-size test) moves keys into
    pages of another size without changing what the definition reads:
    bitwise the same output, with a window, a batch and 16-bit storage."""
    case = W.make_case("relay", seed=41, query_lens=[3, 0, 5], past_lens=[37, 4, 60], num_q_heads=8,
                       num_kv_heads=2, head_dim=16, page_size=8, sliding_window=21)
    moved = W.relayout(case, ps, seed=5)
    assert moved.page_size == ps and moved.block_tables.shape[0] == case.num_seqs
    assert np.array_equal(run_oracle(oracle_mod, moved), run_oracle(oracle_mod, case))
