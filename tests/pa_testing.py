"""Shared test plumbing: move a seeded workload to the GPU, run the library
through its C ABI, and run the oracle on the same storage."""
from __future__ import annotations

import numpy as np

import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

TOL = 2e-3  # max abs error vs the fp64 oracle (bf16 out, fp32 accumulation)

KV_CODE = {"f32": pa.PA_F32, "f16": pa.PA_F16, "bf16": pa.PA_BF16, "u8": pa.PA_U8}


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "u8": torch.uint8}[name]


def to_device(case: W.Case, out_dtype: str | None = None, device="cuda"):
    import torch

    def stored(raw, dt):
        t = torch.from_numpy(np.ascontiguousarray(raw))
        if dt in ("f16", "bf16"):
            t = t.view(torch.int16).view(torch_dtype(dt))
        return t.to(device)

    q = stored(case.q, case.q_dtype)
    if case.kv_dtype == "u8":
        k = torch.from_numpy(case.k_cache).to(device)
        v = torch.from_numpy(case.v_cache).to(device)
    else:
        k = stored(case.k_cache, case.kv_dtype)
        v = stored(case.v_cache, case.kv_dtype)
    od = out_dtype or case.out_dtype
    out = torch.full((case.total_tokens, case.num_q_heads, case.head_dim), float("nan"),
                     dtype=torch_dtype(od), device=device)
    return dict(q=q, k=k, v=v, bt=torch.from_numpy(case.block_tables).to(device),
                pl=torch.from_numpy(case.past_lens).to(device),
                sb=torch.from_numpy(case.subsequence_begins).to(device), out=out)


def dims(case: W.Case, dev) -> pa.PaDims:
    return pa.dims_for(dev["q"], dev["k"], dev["bt"], dev["pl"], dev["out"], num_kv_heads=case.num_kv_heads,
                       page_size=case.page_size, head_dim=case.head_dim)


def run_gpu(case: W.Case, dev=None, out_dtype=None, traced=False, max_context_len=None, workspace=None):
    """Run the verify step on the GPU; returns (out float64 numpy, status bits, trace or None)."""
    import torch
    dev = dev or to_device(case, out_dtype)
    d = dims(case, dev)
    mcl = case.max_context_len if max_context_len is None else max_context_len
    kvc = KV_CODE[case.kv_dtype]
    ws = workspace if workspace is not None else pa.alloc_workspace(d, mcl, case.sliding_window, kvc)
    trace = None
    args = (dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], mcl, case.scale, case.sliding_window, kvc,
            dev["out"], d, ws)
    if traced:
        trace = torch.zeros((case.num_seqs, case.num_kv_heads, case.max_blocks_per_seq), dtype=torch.int32,
                            device=dev["q"].device)
        pa.forward_traced(*args, trace)
    else:
        pa.forward(*args)
    bits = pa.device_status(ws)
    torch.cuda.synchronize()
    out = dev["out"].float().cpu().numpy().astype(np.float64)
    return out, bits, (trace.cpu().numpy() if trace is not None else None)


def run_oracle(case: W.Case, nthreads: int = 0):
    import oracle
    return oracle.forward(case.q, case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                          case.past_lens, case.subsequence_begins, num_q_heads=case.num_q_heads,
                          num_kv_heads=case.num_kv_heads, head_dim=case.head_dim, page_size=case.page_size,
                          num_blocks=case.num_blocks, scale=case.scale, sliding_window=case.sliding_window,
                          nthreads=nthreads)


UNIT_ROUNDOFF = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8, "u8": 2.0 ** -11}


def derived_tolerance(case: W.Case, want, out_dtype=None):
    """Per-element bound for short contexts, where outputs are O(1):
    2e-3 + u_P * sum_j p_j |v_j| / sum_j p_j + u_out * |ref|.
    u_P is the unit roundoff of the softmax weights as the tensor cores consume
    them (the V operand type: bf16 for bf16 caches, f16 for f16 and u8 caches),
    u_out that of the output dtype.  Rounding every weight by at most u_P moves
    the weighted mean by at most u_P * sum p |v| / l; rounding the result moves
    it by at most u_out * |ref|."""
    import test_oracle_pins as P
    kc, vc = P._decode_cache(case)
    q = W.storage_to_f64(case.q, case.q_dtype).reshape(case.total_tokens, case.num_q_heads, case.head_dim)
    G = case.num_q_heads // case.num_kv_heads
    spread = np.zeros_like(want)
    for b in range(case.num_seqs):
        L, t0 = int(case.past_lens[b]), int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            p = L + i
            lo = max(0, p - case.sliding_window + 1) if case.sliding_window > 0 else 0
            js = np.arange(lo, p + 1)
            blk = case.block_tables[b][js // case.page_size]
            for h in range(case.num_q_heads):
                K = kc[blk, h // G, js % case.page_size]
                V = vc[blk, h // G, js % case.page_size]
                s = case.scale * (K @ q[t0 + i, h])
                w = np.exp(s - s.max())
                spread[t0 + i, h] = (w @ np.abs(V)) / w.sum()
    u_p = UNIT_ROUNDOFF[case.kv_dtype]
    u_o = UNIT_ROUNDOFF[out_dtype or case.out_dtype]
    return 2e-3 + u_p * spread + u_o * np.abs(want)


def max_abs_err(got, want):
    assert got.shape == want.shape
    assert np.isfinite(got).all(), f"{np.count_nonzero(~np.isfinite(got))} non-finite outputs"
    return float(np.max(np.abs(got - want))) if got.size else 0.0


def check_parity(case, out_dtype=None, tol=TOL):
    """GPU output and gather trace against the oracle.  tol: the flat 2e-3
    bound for the pages' long-context workloads, or "derived"
    (derived_tolerance) for short-context edge cases whose outputs are O(1),
    where one bf16 rounding alone exceeds 2e-3."""
    got, bits, trace = run_gpu(case, out_dtype=out_dtype, traced=True)
    assert bits == 0, f"device status {bits:#x}"
    want = run_oracle(case)
    err = max_abs_err(got, want)
    if isinstance(tol, str):
        bound = derived_tolerance(case, want, out_dtype)
        worst = float(np.max(np.abs(got - want) - bound))
        assert worst <= 0.0, f"{case.name}: error exceeds the derived bound by {worst:.3e} (max abs {err:.3e})"
    else:
        assert err <= tol, f"{case.name}: max abs err {err:.3e}"
    import oracle
    pages = oracle.pages_touched(case.block_tables, case.past_lens, case.subsequence_begins,
                                 page_size=case.page_size, sliding_window=case.sliding_window)
    for g in range(case.num_kv_heads):
        assert np.array_equal(trace[:, g, :], pages), f"{case.name}: gather trace of KV head {g} differs"
    return err
