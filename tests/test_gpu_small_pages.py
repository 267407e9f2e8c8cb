"""Pages of 1, 2 or 4 tokens on the GPU: the long-context stress layout in
which every key is its own block-table lookup (one token per page), served
by the tensor-memory kernel's cp.async-gather producer (16-bit caches,
head_dim <= 128), the warp-level kernel's per-key bulk copies (16-bit caches,
head_dim 256) and the FFMA kernel (fp32 caches).

Checks: parity with the oracle and a bit-exact gather trace (every page id
a CTA fetched); the same logical K/V in 16-token pages gives bitwise the
same output (the page size only moves keys); the cache update writes 1-token
pages; and a bad block id in a 1-token page sets the status bit."""
import numpy as np
import pytest

import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import KV_CODE, TOL, check_parity, dims, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _expected_kernel(case):
    return 1 if case.kv_dtype == "f32" else (0 if case.head_dim == 256 else 2)


def _kernel(case):
    import torch
    d = dims(case, to_device(case))
    return pa.plan(d, case.max_context_len, case.sliding_window, KV_CODE[case.kv_dtype],
                   torch.cuda.get_device_properties(0).multi_processor_count).kernel


EDGE = {"ps1_batch_edge", "ps1_f32_batch", "ps4_d256_f16_batch", "gemma_swa256_T8_L1500_as_ps2"}

SMALL = [
    lambda: W.long_ctx_b(5000, page_size=1, seed=40),                    # 64 rows
    lambda: W.qwen_gqa(1, 1000, page_size=1, seed=41),                   # 4 rows
    lambda: W.qwen_gqa(4, 1003, page_size=2, seed=42),
    lambda: W.qwen_gqa(4, 20000, page_size=1, seed=43),                  # many partitions, ragged tail
    lambda: W.make_case("ps4_f16", seed=44, query_lens=[3], past_lens=[2047], num_q_heads=16, num_kv_heads=4,
                        head_dim=128, page_size=4, q_dtype="f16", kv_dtype="f16"),
    lambda: W.make_case("ps1_d64_win", seed=45, query_lens=[4], past_lens=[1600], num_q_heads=8, num_kv_heads=2,
                        head_dim=64, page_size=1, sliding_window=300),
    lambda: W.make_case("ps1_batch_edge", seed=46, query_lens=[1, 0, 4, 2, 3], past_lens=[0, 50, 17, 300, 64],
                        num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=1),
    lambda: W.make_case("ps1_f32_batch", seed=47, query_lens=[2, 3], past_lens=[150, 40], num_q_heads=4,
                        num_kv_heads=2, head_dim=128, page_size=1, q_dtype="f32", kv_dtype="f32",
                        sliding_window=33),
    # head_dim 256: unreferenced slots NaN (relayout), ragged last stage
    lambda: W.relayout(W.gemma_hybrid(3001, seed=48), 1, seed=1),
    lambda: W.relayout(W.gemma_hybrid(1500, window=256, T=8, seed=49), 2, seed=2),  # 16 rows, window
    lambda: W.make_case("ps4_d256_f16_batch", seed=57, query_lens=[3, 1, 8, 0], past_lens=[700, 0, 2000, 33],
                        num_q_heads=16, num_kv_heads=4, head_dim=256, page_size=4, q_dtype="f16",
                        kv_dtype="f16"),                                          # 32 rows at T=8
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_small_page_parity(idx):
    case = SMALL[idx]()
    assert _kernel(case) == _expected_kernel(case)
    check_parity(case, tol="derived" if case.name in EDGE else TOL)


FULL = [
    lambda: W.long_ctx_b(131072, page_size=1),
    lambda: W.long_ctx_b(184320, page_size=1),
    lambda: W.qwen_gqa(4, 32768, page_size=1),
    lambda: W.relayout(W.gemma_hybrid(32768), 1, seed=3),
]


@pytest.mark.slow
@pytest.mark.parametrize("idx", range(len(FULL)))
def test_small_page_parity_full_size(idx):
    check_parity(FULL[idx]())


@pytest.mark.parametrize("make,ps", [
    (lambda: W.qwen_gqa(4, 20000, seed=50), 1),
    (lambda: W.long_ctx_b(9000, seed=51), 2),
    (lambda: W.make_case("d64_f16", seed=52, query_lens=[8], past_lens=[3000], num_q_heads=8, num_kv_heads=2,
                         head_dim=64, page_size=16, q_dtype="f16", kv_dtype="f16"), 4),
])
def test_page_size_does_not_change_the_output(make, ps):
    """16-token pages (TMA boxes) and 1-4-token pages (cp.async gather) of the
    same logical K/V: the same partitions and the same arithmetic, so the
    outputs agree bit for bit."""
    case = make()
    small = W.relayout(case, ps, seed=7)
    assert _kernel(case) == 2 and _kernel(small) == 2
    a, bits_a, _ = run_gpu(case)
    b, bits_b, _ = run_gpu(small)
    assert bits_a == 0 and bits_b == 0
    assert np.array_equal(a, b)


@pytest.mark.parametrize("ps", [1, 2, 4])
def test_head_dim_256_page_size_does_not_change_the_output(ps):
    """head_dim 256: 8-token pages (TMA boxes) and 1-4-token pages (one bulk
    copy per key row) of the same logical K/V take the same partitions and
    arithmetic, so the outputs agree bit for bit."""
    case = W.gemma_hybrid(5000, T=4, seed=58)
    a_case = W.relayout(case, 8, seed=9)
    b_case = W.relayout(case, ps, seed=10)
    da, db = dims(a_case, to_device(a_case)), dims(b_case, to_device(b_case))
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pa_, pb_ = (pa.plan(d, c.max_context_len, 0, KV_CODE[c.kv_dtype], sms) for d, c in ((da, a_case), (db, b_case)))
    assert pa_.kernel == 0 and pb_.kernel == 0
    assert (pa_.num_partitions, pa_.part_tokens) == (pb_.num_partitions, pb_.part_tokens)
    a, bits_a, _ = run_gpu(a_case)
    b, bits_b, _ = run_gpu(b_case)
    assert bits_a == 0 and bits_b == 0
    assert np.array_equal(a, b)


def test_cache_update_into_one_token_pages():
    import torch
    import oracle
    case = W.qwen_gqa(3, 700, page_size=1, seed=53)
    kn, vn = W.new_tokens(case, "bf16", seed=5)
    want_k, want_v = oracle.cache_update(kn, vn, "bf16", case.k_cache, case.v_cache, case.kv_dtype,
                                         case.block_tables, case.past_lens, case.subsequence_begins,
                                         num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                                         page_size=case.page_size, num_blocks=case.num_blocks)
    dev = to_device(case)
    d = dims(case, dev)
    src = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.bfloat16).cuda()
    pa.cache_update(src(kn), src(vn), dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], d)
    torch.cuda.synchronize()
    assert np.array_equal(dev["k"].cpu().view(torch.int16).numpy().view(np.uint8),
                          np.ascontiguousarray(want_k).view(np.uint8))
    assert np.array_equal(dev["v"].cpu().view(torch.int16).numpy().view(np.uint8),
                          np.ascontiguousarray(want_v).view(np.uint8))


@pytest.mark.parametrize("make", [
    lambda: W.qwen_gqa(4, 3000, page_size=1, seed=54),
    lambda: W.relayout(W.gemma_hybrid(3000, seed=59), 1, seed=4),
])
def test_bad_block_id_in_a_one_token_page_sets_the_status(make):
    case = make()
    bt = case.block_tables.copy()
    bt[0, 1234] = case.num_blocks + 5
    bad = W.Case(**{**case.__dict__, "block_tables": bt})
    got, bits, _ = run_gpu(bad)
    assert bits & 0x4  # PA_STATUS_BLOCK_ID
    # the sequence's rows are zero (the partition holding the bad id poisons them)
    assert np.all(got == 0.0)


@pytest.mark.parametrize("make", [
    lambda: W.long_ctx_b(3000, page_size=1, seed=55),
    lambda: W.make_case("ps2_tree_batch_win", seed=56, query_lens=[5, 0, 8, 3], past_lens=[900, 10, 1300, 40],
                        num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=2, sliding_window=400),
    lambda: W.relayout(W.gemma_hybrid(2500, T=8, seed=60), 1, seed=5),
])
def test_tree_mask_on_small_pages(make):
    import oracle
    from test_gpu_tree import _gpu_tree, random_tree_masks
    from pa_testing import derived_tolerance
    case = make()
    mask = random_tree_masks(case, seed=3)
    want = oracle.forward(case.q, case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                          case.past_lens, case.subsequence_begins, num_q_heads=case.num_q_heads,
                          num_kv_heads=case.num_kv_heads, head_dim=case.head_dim, page_size=case.page_size,
                          num_blocks=case.num_blocks, scale=case.scale, sliding_window=case.sliding_window,
                          tree_mask=mask)
    got, bits, k, _ = _gpu_tree(case, mask)
    assert bits == 0 and k == _expected_kernel(case)
    if case.sliding_window:  # short windows: O(1) outputs, the derived bound
        assert float(np.max(np.abs(got - want) - derived_tolerance(case, want))) <= 0.0
    else:
        assert float(np.max(np.abs(got - want))) <= TOL
