"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance: max abs error <= 2e-3 (bf16 / f16 output, fp32 accumulation);
gather traces bit-exact.  Reduced-size cases span several pipeline stages,
several partitions and ragged tails; the full-size cases are the five
workload families at their stated sizes.
"""
import numpy as np
import pytest

from paged_attention_speculative_gb300 import workloads as W

from pa_testing import TOL, check_parity as _check, run_gpu, to_device

pytestmark = pytest.mark.gpu


EDGE = {"batch_edge", "window1", "f32_win_batch"}

SMALL = [
    lambda: W.tiny(),
    lambda: W.qwen_gqa(1, 1000, seed=1),
    lambda: W.qwen_gqa(2, 1003, seed=2),
    lambda: W.qwen_gqa(3, 2047, seed=3),
    lambda: W.qwen_gqa(4, 777, seed=4),
    lambda: W.qwen_u8(1, 1500, seed=5),
    lambda: W.qwen_u8(3, 1234, seed=6),
    lambda: W.qwen_u8(6, 2345, seed=15),   # 24 rows: the u8 keys-on-M kernel by default
    lambda: W.make_case("u8_batch_t8", seed=16, query_lens=[8, 5, 0, 7], past_lens=[1900, 700, 20, 2500],
                        num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, kv_dtype="u8"),
    lambda: W.gemma_hybrid(1500, seed=7),
    lambda: W.gemma_hybrid(3000, window=1024, seed=8),
    lambda: W.batched_mix_a(seed=9),
    lambda: W.long_ctx_b(5000, seed=10),
    lambda: W.make_case("f16_gqa", seed=11, query_lens=[3], past_lens=[900], num_q_heads=16, num_kv_heads=4,
                        head_dim=128, page_size=32, q_dtype="f16", kv_dtype="f16"),
    lambda: W.make_case("d64_bf16", seed=12, query_lens=[4], past_lens=[600], num_q_heads=8, num_kv_heads=2,
                        head_dim=64, page_size=16),
    lambda: W.make_case("u8_d256_win", seed=13, query_lens=[2], past_lens=[2100], num_q_heads=8, num_kv_heads=4,
                        head_dim=256, page_size=64, kv_dtype="u8", q_dtype="f16", sliding_window=700),
    lambda: W.make_case("u8_t8_g8", seed=14, query_lens=[8], past_lens=[1100], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=16, kv_dtype="u8"),
    lambda: W.make_case("batch_edge", seed=15, query_lens=[1, 0, 4, 2, 3], past_lens=[0, 50, 17, 300, 64],
                        num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=8),
    lambda: W.make_case("f32_win_batch", seed=16, query_lens=[2, 3], past_lens=[150, 40], num_q_heads=4,
                        num_kv_heads=2, head_dim=128, page_size=16, q_dtype="f32", kv_dtype="f32",
                        sliding_window=33),
    lambda: W.make_case("d256_rows16", seed=18, query_lens=[8], past_lens=[1500], num_q_heads=32, num_kv_heads=16,
                        head_dim=256, page_size=64),
    lambda: W.make_case("rows32_u8", seed=19, query_lens=[8], past_lens=[2500], num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=16, kv_dtype="u8"),
    lambda: W.make_case("window1", seed=17, query_lens=[4], past_lens=[200], num_q_heads=8, num_kv_heads=2,
                        head_dim=128, page_size=16, sliding_window=1),
    # odd numbers of output rows (the combine packs two rows per CTA; its last
    # CTA then has one row past the end), on each partition kernel
    lambda: W.make_case("odd_rows_tc", seed=21, query_lens=[3], past_lens=[3000], num_q_heads=5, num_kv_heads=1,
                        head_dim=128, page_size=16),
    lambda: W.make_case("odd_rows_u8", seed=22, query_lens=[5], past_lens=[2600], num_q_heads=3, num_kv_heads=1,
                        head_dim=128, page_size=16, kv_dtype="u8"),
    lambda: W.make_case("odd_rows_d256", seed=23, query_lens=[3, 1], past_lens=[2200, 1700], num_q_heads=3,
                        num_kv_heads=1, head_dim=256, page_size=64),
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_parity_reduced(idx):
    case = SMALL[idx]()
    _check(case, tol="derived" if case.name in EDGE else TOL)


@pytest.mark.parametrize("out_dtype", ["f32", "f16"])
def test_parity_other_out_dtypes(out_dtype):
    _check(W.qwen_gqa(3, 1500, seed=20), out_dtype=out_dtype)


FULL = [
    lambda: W.tiny(),
    lambda: W.qwen_gqa(1, 8192), lambda: W.qwen_gqa(4, 8192), lambda: W.qwen_gqa(2, 32768),
    lambda: W.qwen_gqa(4, 32768),
    lambda: W.qwen_u8(1, 32768), lambda: W.qwen_u8(3, 65536), lambda: W.qwen_u8(8, 32768),
    lambda: W.gemma_hybrid(32768), lambda: W.gemma_hybrid(51200), lambda: W.gemma_hybrid(32768, window=1024),
    lambda: W.batched_mix_a(),
    lambda: W.long_ctx_b(131072), lambda: W.long_ctx_b(184320),
]


@pytest.mark.slow
@pytest.mark.parametrize("idx", range(len(FULL)))
def test_parity_full_size(idx):
    _check(FULL[idx]())


def test_t_tokens_equal_t_single_token_decodes():
    """The pages' equivalence, on the GPU: a T-token verify equals T
    single-token decodes with past_len L, L+1, ... (within tolerance)."""
    case = W.qwen_gqa(4, 3000, seed=30)
    multi, bits, _ = run_gpu(case)
    assert bits == 0
    for i in range(4):
        single = W.Case(**{**case.__dict__, "q": case.q[i:i + 1].copy(),
                           "past_lens": np.array([3000 + i], np.int32),
                           "subsequence_begins": np.array([0, 1], np.int32), "name": f"single{i}"})
        got, bits, _ = run_gpu(single)
        assert bits == 0
        assert np.max(np.abs(got[0] - multi[i])) <= TOL


def test_block_table_permutation_is_bitwise_invariant():
    case = W.qwen_gqa(3, 2500, seed=31)
    a, _, _ = run_gpu(case)
    rng = np.random.default_rng(5)
    perm = rng.permutation(case.num_blocks)
    inv = np.argsort(perm)
    moved = W.Case(**{**case.__dict__, "k_cache": case.k_cache[inv].copy(), "v_cache": case.v_cache[inv].copy(),
                      "block_tables": perm[case.block_tables].astype(np.int32)})
    b, _, _ = run_gpu(moved)
    assert np.array_equal(a, b)


def test_deterministic_across_calls():
    case = W.qwen_u8(3, 4000, seed=32)
    dev = to_device(case)
    a, _, _ = run_gpu(case, dev=dev)
    b, _, _ = run_gpu(case, dev=dev)
    assert np.array_equal(a, b)


def test_future_keys_do_not_leak():
    """Changing the last new token's K/V moves only that token's output."""
    case = W.qwen_gqa(4, 1000, seed=33)
    a, _, _ = run_gpu(case)
    k = case.k_cache.copy()
    v = case.v_cache.copy()
    p = 1003
    blk = case.block_tables[0][p // 16]
    k[blk, :, p % 16] = W.to_storage(np.full((8, 128), 3.0, np.float32), "bf16")
    v[blk, :, p % 16] = W.to_storage(np.full((8, 128), -2.0, np.float32), "bf16")
    b, _, _ = run_gpu(W.Case(**{**case.__dict__, "k_cache": k, "v_cache": v}))
    assert np.array_equal(a[:3], b[:3])
    assert not np.array_equal(a[3], b[3])
