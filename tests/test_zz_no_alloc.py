"""pa_verify_forward_no_alloc: the entry point for callers that cannot
allocate device memory (for example a C-only host whose GPU memory is held by
another runtime's pool, or a serving loop that must not call cudaMalloc once
it runs).  Its split-KV partials live in a fixed 16 MiB array inside the
library instead of a caller-provided workspace.

Checked through the C ABI against pa_verify_forward on two calls in a row,
and for its size limit.  Kept in a file collected last so that a run stopping
at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import KV_CODE, TOL, dims, run_gpu, to_device

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


@pytest.mark.parametrize("pair", [0, 1])
def test_two_calls_in_a_row_match_the_workspace_entry_point(pair):
    cases = [
        [W.qwen_gqa(4, 3000, seed=60), W.qwen_u8(3, 2200, seed=61)],
        [W.gemma_hybrid(2500, window=1024, seed=62), W.long_ctx_b(4000, seed=63)],
    ][pair]
    for case in cases:  # two calls in a row on the shared scratch
        want, bits, _ = run_gpu(case)  # pa_verify_forward with its own workspace
        assert bits == 0
        dev = to_device(case)
        assert _no_alloc(case, dev) == 0
        got = dev["out"].float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert float(np.max(np.abs(got - want))) <= TOL


def test_rejects_calls_that_need_more_than_the_scratch():
    import torch
    # A valid problem whose planned partials (64 query rows x ~120 partitions
    # x 520 bytes per row) exceed 16 MiB: max_context_len sizes the grid.
    case = W.make_case("big_plan", seed=64, query_lens=[8], past_lens=[100], num_q_heads=64, num_kv_heads=8,
                       head_dim=128, page_size=16, table_slack=125_000, poison=False)
    dev = to_device(case)
    dev["out"].fill_(7.0)
    rc = _no_alloc(case, dev, max_context_len=2_000_000)
    assert rc == -7, pa.status_string(rc)
    assert bool((dev["out"] == 7.0).all())
