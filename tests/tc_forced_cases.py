"""Run in a child process with PA_VERIFY_KERNEL=tc (the 16-bit rows-on-M
tensor-memory kernel wherever it applies), PA_VERIFY_KERNEL=mma (the
warp-level kernel for 16-bit and u8 caches) or neither (the default choice,
e.g. with a forced partition size): prints one JSON line per case with the
plan's kernel, the max abs error against the oracle and the gather-trace
check."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from paged_attention_speculative_gb300 import workloads as W  # noqa: E402
import paged_attention_speculative_gb300 as pa  # noqa: E402
from pa_testing import KV_CODE, derived_tolerance, dims, max_abs_err, run_gpu, run_oracle, to_device  # noqa: E402

EDGE = {"tc_window_batch"}  # short contexts (O(1) outputs): derived bf16 bound

CASES = [
    lambda: W.qwen_gqa(1, 1000, seed=71),
    lambda: W.qwen_gqa(4, 2047, seed=72),
    lambda: W.long_ctx_b(3000, seed=73),
    lambda: W.make_case("tc_f16_rows40", seed=74, query_lens=[5], past_lens=[1777], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=32, q_dtype="f16", kv_dtype="f16"),
    lambda: W.make_case("tc_d64_rows64", seed=75, query_lens=[8], past_lens=[900], num_q_heads=32, num_kv_heads=4,
                        head_dim=64, page_size=16),
    lambda: W.make_case("tc_window_batch", seed=76, query_lens=[8, 3, 0, 6], past_lens=[1200, 64, 10, 333],
                        num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=16, sliding_window=300),
    lambda: W.make_case("tc_ps64_rows64", seed=78, query_lens=[8], past_lens=[2000], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=64),
    lambda: W.qwen_u8(1, 1500, seed=79),
    lambda: W.qwen_u8(3, 2345, seed=80),
    lambda: W.make_case("u8_rows64_f16q", seed=81, query_lens=[8], past_lens=[3100], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=16, kv_dtype="u8", q_dtype="f16"),
    lambda: W.make_case("u8_window_ps32", seed=82, query_lens=[4, 2], past_lens=[1500, 700], num_q_heads=32,
                        num_kv_heads=8, head_dim=128, page_size=32, kv_dtype="u8", sliding_window=500),
    lambda: W.make_case("tc_ps8_long", seed=77, query_lens=[7], past_lens=[9000], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=8),
]

if __name__ == "__main__":
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for make in CASES:
        case = make()
        plan = pa.plan(dims(case, to_device(case)), case.max_context_len, case.sliding_window, KV_CODE[case.kv_dtype],
                       sms)
        got, bits, trace = run_gpu(case, traced=True)
        want = run_oracle(case)
        pages = oracle.pages_touched(case.block_tables, case.past_lens, case.subsequence_begins,
                                     page_size=case.page_size, sliding_window=case.sliding_window)
        trace_ok = all(np.array_equal(trace[:, g, :], pages) for g in range(case.num_kv_heads))
        excess = None
        if case.name in EDGE:
            excess = float(np.max(np.abs(got - want) - derived_tolerance(case, want)))
        print(json.dumps({"case": case.name, "kernel": plan.kernel, "bits": bits, "err": max_abs_err(got, want), "excess": excess,
                          "trace_ok": trace_ok}), flush=True)
