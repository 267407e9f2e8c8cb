"""pa_verify_forward_no_alloc: the entry point for callers that cannot
allocate device memory (for example a C-only host whose GPU memory is held by
another runtime's pool, or a serving loop that must not call cudaMalloc once
it runs).  Its split-KV partials live in a fixed 16 MiB array inside the
library instead of a caller-provided workspace.

Checked through the C ABI on calls in a row: bit for bit against
pa_verify_forward (same plan, same kernels), and against the fp64 oracle
within the flat tolerance.  Also: a call with few partitions right after one
with many (stale partials in the shared array would show), a call whose
block table is bad followed by a clean one (its zeroed rows and status must
not leak), and the size limit.  Kept in a file collected last so that a run
stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import KV_CODE, TOL, dims, max_abs_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def _no_alloc(case, dev, max_context_len=None):
    import torch
    lib = pa.load_library()
    d = dims(case, dev)
    mcl = case.max_context_len if max_context_len is None else max_context_len
    stream = torch.cuda.current_stream()
    rc = lib.pa_verify_forward_no_alloc(
        ctypes.c_void_p(dev["q"].data_ptr()), ctypes.c_void_p(dev["k"].data_ptr()),
        ctypes.c_void_p(dev["v"].data_ptr()), ctypes.c_void_p(dev["bt"].data_ptr()),
        ctypes.c_void_p(dev["pl"].data_ptr()), ctypes.c_void_p(dev["sb"].data_ptr()), int(mcl),
        float(case.scale), int(case.sliding_window), int(KV_CODE[case.kv_dtype]),
        ctypes.c_void_p(dev["out"].data_ptr()), ctypes.byref(d), ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    return rc


def _out(dev):
    return dev["out"].float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("pair", [0, 1])
def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle(pair):
    cases = [
        [W.qwen_gqa(4, 3000, seed=60), W.qwen_u8(3, 2200, seed=61)],
        [W.gemma_hybrid(2500, window=1024, seed=62), W.long_ctx_b(4000, seed=63)],
    ][pair]
    for case in cases:  # two calls in a row on the shared scratch
        want, bits, _ = run_gpu(case)  # pa_verify_forward with its own workspace
        assert bits == 0
        dev = to_device(case)
        assert _no_alloc(case, dev) == 0
        got = _out(dev)
        assert np.array_equal(got, want), "same plan and kernels: the outputs must match bit for bit"
        assert max_abs_err(got, run_oracle(case)) <= TOL


def test_few_partitions_after_many():
    """A call planned with many partitions leaves partials all over the shared
    array; the next call, with few partitions and the same dims, must read
    only its own."""
    big = W.qwen_gqa(2, 20000, seed=64)  # 19 partitions of ~1k keys, 64 query rows
    dev_big = to_device(big)
    assert _no_alloc(big, dev_big) == 0
    small = W.qwen_gqa(4, 3000, seed=65)  # fewer partitions, 128 query rows
    want, bits, _ = run_gpu(small)
    assert bits == 0
    dev = to_device(small)
    assert _no_alloc(small, dev) == 0
    assert np.array_equal(_out(dev), want)


def test_bad_call_then_clean_call():
    """A block id outside the pool: the call leaves its rows zero; the next
    clean call is unaffected (its status word was cleared, its rows are
    computed)."""
    bad = W.qwen_gqa(2, 1500, seed=66)
    bt = bad.block_tables.copy()
    bt[0, 5] = bad.num_blocks + 7
    bad = W.Case(**{**bad.__dict__, "block_tables": bt})
    dev_bad = to_device(bad)
    assert _no_alloc(bad, dev_bad) == 0
    assert float(np.max(np.abs(_out(dev_bad)))) == 0.0
    clean = W.qwen_gqa(2, 1500, seed=67)
    want, bits, _ = run_gpu(clean)
    assert bits == 0
    dev = to_device(clean)
    assert _no_alloc(clean, dev) == 0
    assert np.array_equal(_out(dev), want)


def test_rejects_calls_that_need_more_than_the_scratch():
    # A valid problem whose planned partials (64 query rows x ~120 partitions
    # x 520 bytes per row) exceed 16 MiB: max_context_len sizes the grid.
    case = W.make_case("big_plan", seed=68, query_lens=[8], past_lens=[100], num_q_heads=64, num_kv_heads=8,
                       head_dim=128, page_size=16, table_slack=125_000, poison=False)
    dev = to_device(case)
    dev["out"].fill_(7.0)
    rc = _no_alloc(case, dev, max_context_len=2_000_000)
    assert rc == -7, pa.status_string(rc)
    assert bool((dev["out"] == 7.0).all())
