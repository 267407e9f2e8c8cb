"""Device-detected errors set status bits, skip work and leave rows zero;
nothing traps.  (All inputs here are in-bounds for every memory access: the
kernels validate block ids before use and TMA bounds-checks the tiles.)"""
import numpy as np
import pytest

from paged_attention_speculative_gb300 import workloads as W

from pa_testing import run_gpu

pytestmark = pytest.mark.gpu


def test_bad_block_id_sets_status_and_zeroes_rows():
    case = W.qwen_gqa(2, 3000, seed=40)
    case.block_tables[0, 5] = case.num_blocks + 7
    out, bits, _ = run_gpu(case)
    assert bits & 0x4
    assert np.all(out == 0.0)


def test_negative_block_id_sets_status():
    case = W.qwen_gqa(1, 500, seed=41)
    case.block_tables[0, 2] = -3
    out, bits, _ = run_gpu(case)
    assert bits & 0x4
    assert np.all(out == 0.0)


def test_context_longer_than_max_context_len():
    case = W.qwen_gqa(3, 2000, seed=42)
    out, bits, _ = run_gpu(case, max_context_len=1500)
    assert bits & 0x2
    assert np.all(out == 0.0)


def test_query_len_above_eight_is_reported():
    case = W.make_case("t9", seed=43, query_lens=[9], past_lens=[100], num_q_heads=4, num_kv_heads=4,
                       head_dim=128, page_size=16)
    out, bits, _ = run_gpu(case)
    assert bits & 0x1
    assert np.all(out == 0.0)


def test_other_sequences_unaffected_by_a_bad_one():
    case = W.make_case("mixed_bad", seed=44, query_lens=[2, 3], past_lens=[400, 700], num_q_heads=8,
                       num_kv_heads=2, head_dim=128, page_size=16)
    good, bits, _ = run_gpu(case)
    assert bits == 0
    case.block_tables[0, 3] = -1
    out, bits, _ = run_gpu(case)
    assert bits & 0x4
    assert np.all(out[:2] == 0.0)
    assert np.array_equal(out[2:], good[2:])
