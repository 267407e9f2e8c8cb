#!/usr/bin/env python
"""bench.py — µs per verify step and KV-read HBM GB/s of paged verify attention.

Headline workload: Qwen-like GQA verify (batch 1, 32 query / 8 KV heads,
head_dim 128, page 16, bf16) with T=4 new query tokens at past_len 32768.
One step = one pa_verify_forward (split-KV partition kernel + per-token LSE
combine) over that batch.  `value` = algorithmic KV-read bytes per step /
device time per step (GB/s).  Steps are replayed from a CUDA graph, rotating
over KV-cache replicas whose total exceeds 2x the L2 cache, so every step
streams its KV from HBM.

Also printed (same JSON line): the partition kernel's roofline against the
measured HBM copy rate, an end-to-end figure through host buffers, the fp64
oracle timed on the host cores, the clocks seen while timing, and a sweep of
all workload families (µs/step, KV GB/s, fraction of the roofline, ratio to
T=1 at the same context).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = dict(name="qwen_gqa_T4_L32768", Hq=32, Hkv=8, D=128, ps=16, kv="bf16", q_lens=[4], past=[32768], window=0)

SWEEP = [
    dict(name="qwen_gqa_T{T}_L{L}", Hq=32, Hkv=8, D=128, ps=16, kv="bf16", T=[1, 2, 3, 4], L=[8192, 32768], window=0),
    dict(name="qwen_u8_T{T}_L{L}", Hq=32, Hkv=8, D=128, ps=16, kv="u8", T=[1, 3, 8], L=[32768, 65536], window=0),
    dict(name="gemma_global_T{T}_L{L}", Hq=32, Hkv=16, D=256, ps=64, kv="bf16", T=[1, 2], L=[32768, 51200], window=0),
    dict(name="gemma_swa1024_T{T}_L{L}", Hq=32, Hkv=16, D=256, ps=64, kv="bf16", T=[1, 2], L=[32768], window=1024),
    dict(name="long_T{T}_L{L}", Hq=64, Hkv=8, D=128, ps=16, kv="bf16", T=[1, 8], L=[131072, 184320], window=0),
]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# Device-side synthetic workload (same shapes and distributions as the seeded
# recipe used by the tests: N(0,1) rounded once to the cache dtype, u8 by
# per-token min/max quantisation, a seeded random page permutation).  Only the
# pages some query reads get physical blocks; every replica gets its own.
# ---------------------------------------------------------------------------
class DeviceWorkload:
    def __init__(self, Hq, Hkv, D, ps, kv, q_lens, past, window, min_bytes, seed=0, max_replicas=64):
        import torch
        import paged_attention_speculative_gb300 as pa
        self.Hq, self.Hkv, self.D, self.ps, self.kv, self.window = Hq, Hkv, D, ps, kv, window
        self.q_lens, self.past = list(q_lens), list(past)
        B = len(past)
        self.B = B
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.T_total = sum(q_lens)
        self.max_ctx = max(L + T for L, T in zip(past, q_lens))
        self.max_blocks = (self.max_ctx + ps - 1) // ps
        read_pages = []
        for L, T in zip(past, q_lens):
            khi = L + T - 1
            klo = max(0, L - window + 1) if window > 0 else 0
            read_pages.append(list(range(klo // ps, khi // ps + 1)))
        n_read = sum(len(r) for r in read_pages)
        eb = 1 if kv == "u8" else 2
        page_bytes = ps * (D + 4) if kv == "u8" else ps * D * eb
        bytes_per_replica = 2 * n_read * Hkv * page_bytes
        self.replicas = max(2, min(max_replicas, math.ceil(min_bytes / bytes_per_replica)))
        nb = 1 + self.replicas * n_read
        self.num_blocks = nb
        perm = torch.randperm(nb - 1, generator=g) + 1
        bts = torch.zeros((self.replicas, B, self.max_blocks), dtype=torch.int32)
        cur = 0
        for r in range(self.replicas):
            for b in range(B):
                n = len(read_pages[b])
                bts[r, b, read_pages[b][0]: read_pages[b][0] + n] = perm[cur: cur + n].to(torch.int32)
                cur += n
        self.block_tables = bts.cuda()
        self.block_tables_host = bts.pin_memory()
        gd = torch.Generator(device="cuda").manual_seed(seed + 1)
        qdt = torch.bfloat16
        self.q = torch.randn((self.T_total, Hq, D), generator=gd, device="cuda").to(qdt)
        if kv == "u8":
            self.k = self._u8_pool(nb, gd)
            self.v = self._u8_pool(nb, gd, dim_major=True)  # V records hold their codes dim-major
        else:
            dt = torch.bfloat16 if kv == "bf16" else torch.float16
            self.k = torch.randn((nb, Hkv, ps, D), generator=gd, device="cuda").to(dt)
            self.v = torch.randn((nb, Hkv, ps, D), generator=gd, device="cuda").to(dt)
        self.past_lens = torch.tensor(past, dtype=torch.int32, device="cuda")
        begins = [0]
        for T in q_lens:
            begins.append(begins[-1] + T)
        self.begins = torch.tensor(begins, dtype=torch.int32, device="cuda")
        self.out = torch.empty((self.T_total, Hq, D), dtype=qdt, device="cuda")
        self.kv_code = {"bf16": pa.PA_BF16, "f16": pa.PA_F16, "u8": pa.PA_U8}[kv]
        self.dims = pa.dims_for(self.q, self.k, self.block_tables[0], self.past_lens, self.out, num_kv_heads=Hkv,
                                page_size=ps, head_dim=D)
        self.ws = pa.alloc_workspace(self.dims, self.max_ctx, window, self.kv_code)
        self.scale = 1.0 / math.sqrt(D)
        # algorithmic bytes / flops of one step
        n_keys = [min(L + T, window + T - 1) if window > 0 else L + T for L, T in zip(past, q_lens)]
        per_key = 2 * D * eb + (8 if kv == "u8" else 0)
        self.kv_bytes = sum(n_keys) * Hkv * per_key
        G = Hq // Hkv
        vis = 0
        for L, T in zip(past, q_lens):
            for i in range(T):
                p = L + i
                lo = max(0, p - window + 1) if window > 0 else 0
                vis += p - lo + 1
        self.flops = 4 * D * G * Hkv * vis
        self.total_device_bytes = sum(t.numel() * t.element_size() for t in (self.k, self.v))
        # the new tokens' K / V for the cache update (bf16, like a projection's output)
        self.k_new = torch.randn((self.T_total, Hkv, D), generator=gd, device="cuda").to(torch.bfloat16)
        self.v_new = torch.randn((self.T_total, Hkv, D), generator=gd, device="cuda").to(torch.bfloat16)
        # bytes one update moves: both new-token tensors read, their slots written
        slot_bytes = D + 4 if kv == "u8" else D * eb
        self.update_bytes = 2 * self.T_total * Hkv * (D * 2 + slot_bytes)

    def _u8_pool(self, nb, gd, dim_major=False):
        import torch
        x = torch.randn((nb, self.Hkv, self.ps, self.D), generator=gd, device="cuda")
        mn = x.amin(dim=-1)
        mx = x.amax(dim=-1)
        scale = ((mx - mn) / 255.0)
        scale = torch.where(scale > 0, scale, torch.ones_like(scale)).half()
        s = scale.float()
        zp = torch.clamp(torch.round(-mn / s), 0, 255)
        codes = torch.clamp(torch.round(x / s[..., None] + zp[..., None]), 0, 255).to(torch.uint8)
        ps, D = self.ps, self.D
        rec = torch.empty((nb, self.Hkv, ps * (D + 4)), dtype=torch.uint8, device="cuda")
        c = codes.transpose(2, 3) if dim_major else codes
        rec[:, :, : ps * D] = c.contiguous().reshape(nb, self.Hkv, ps * D)
        rec[:, :, ps * D: ps * D + 2 * ps] = scale.contiguous().view(torch.uint8).reshape(nb, self.Hkv, 2 * ps)
        rec[:, :, ps * D + 2 * ps:] = zp.half().contiguous().view(torch.uint8).reshape(nb, self.Hkv, 2 * ps)
        return rec

    def forward(self, r, stream=None):
        import paged_attention_speculative_gb300 as pa
        pa.forward(self.q, self.k, self.v, self.block_tables[r], self.past_lens, self.begins, self.max_ctx,
                   self.scale, self.window, self.kv_code, self.out, self.dims, self.ws, stream=stream)

    def partition(self, r, stream=None):
        import paged_attention_speculative_gb300 as pa
        pa.partition(self.q, self.k, self.v, self.block_tables[r], self.past_lens, self.begins, self.max_ctx,
                     self.scale, self.window, self.kv_code, self.out, self.dims, self.ws, stream=stream)

    def forward_tree(self, r, tree_mask, stream=None):
        import paged_attention_speculative_gb300 as pa
        pa.forward_tree(self.q, self.k, self.v, self.block_tables[r], self.past_lens, self.begins, self.max_ctx,
                        self.scale, self.window, self.kv_code, self.out, self.dims, self.ws, tree_mask,
                        stream=stream)

    def forward_mixed(self, r, stream=None):
        import paged_attention_speculative_gb300 as pa
        if not hasattr(self, "ws_mixed"):
            self.ws_mixed = pa.alloc_mixed_workspace(self.dims, self.max_ctx, self.window, self.kv_code)
        pa.forward_mixed(self.q, self.k, self.v, self.block_tables[r], self.past_lens, self.begins, self.max_ctx,
                         self.scale, self.window, self.kv_code, self.out, self.dims, self.ws_mixed, stream=stream)

    def cache_update(self, r, stream=None):
        import paged_attention_speculative_gb300 as pa
        pa.cache_update(self.k_new, self.v_new, self.k, self.v, self.block_tables[r], self.past_lens, self.begins,
                        self.dims, stream=stream)

    def combine(self, stream=None):
        import paged_attention_speculative_gb300 as pa
        pa.combine(self.past_lens, self.begins, self.max_ctx, self.window, self.kv_code, self.out, self.dims,
                   self.ws, stream=stream)

    def plan(self):
        import paged_attention_speculative_gb300 as pa
        import torch
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        return pa.plan(self.dims, self.max_ctx, self.window, self.kv_code, sms)

    def launches_per_step(self):
        return 1 + (1 if self.plan().num_partitions > 1 else 0)


def mixed_sweep(stream, hbm_peak, l2):
    """Verify steps and prefill chunks in one pa_forward_mixed call, against
    each part alone (verify steps: pa_forward_mixed with no chunk, which is
    the verify path; chunks: pa_forward_mixed with no verify step)."""
    import torch
    tc_peak = peaks().get("bf16_tflops", 1900.0)
    rows = []
    for name, hq, hkv, d, vq, vl, pq, plen in (
            ("qwen_4xT4_L32768+T512_L32768", 32, 8, 128, [4] * 4, [32768] * 4, [512], [32768]),
            ("qwen_4xT4_L32768+T2048_L0", 32, 8, 128, [4] * 4, [32768] * 4, [2048], [0]),
            ("long_T8_L131072+T256_L131072", 64, 8, 128, [8], [131072], [256], [131072]),
            ("qwen_4xT4_L32768+T64_L32768", 32, 8, 128, [4] * 4, [32768] * 4, [64], [32768])):
        us = {}
        for part, ql, pl in (("mixed", vq + pq, vl + plen), ("verify", vq, vl), ("prefill", pq, plen)):
            w = DeviceWorkload(hq, hkv, d, 16, "bf16", ql, pl, 0, min_bytes=2 * l2, seed=17)
            us[part] = time_calls(lambda r: w.forward_mixed(r, stream), w.replicas, stream, reps=16, trials=10)
            if part == "prefill":
                pf_flops = w.flops
            del w
            torch.cuda.empty_cache()
        rows.append({"workload": name, "mixed_us": round(us["mixed"], 2), "verify_alone_us": round(us["verify"], 2),
                     "prefill_alone_us": round(us["prefill"], 2),
                     "mixed_vs_sum": round(us["mixed"] / (us["verify"] + us["prefill"]), 3),
                     "prefill_tflops": round(pf_flops / (us["prefill"] * 1e-6) / 1e12, 1),
                     "prefill_frac_of_measured_bf16": round(pf_flops / (us["prefill"] * 1e-6) / 1e12 / tc_peak, 3)})
        log(f"[bench] mixed {rows[-1]}")
    return rows


def small_page_sweep(stream, hbm_peak, l2):
    """The same verify step with the cache in 16-token (head_dim 256: 64-token)
    pages and in 1-, 2- or 4-token pages (one block-table lookup per key at
    page size 1)."""
    import torch
    rows = []
    for name, hq, hkv, d, T, L, sizes in (("long_T8_L131072", 64, 8, 128, 8, 131072, (16, 4, 2, 1)),
                                          ("long_T8_L184320", 64, 8, 128, 8, 184320, (16, 1)),
                                          ("qwen_gqa_T4_L32768", 32, 8, 128, 4, 32768, (16, 1)),
                                          ("qwen_gqa_T1_L32768", 32, 8, 128, 1, 32768, (16, 1)),
                                          ("gemma_global_T2_L32768", 32, 16, 256, 2, 32768, (64, 4, 1))):
        base = None
        for ps in sizes:
            w = DeviceWorkload(hq, hkv, d, ps, "bf16", [T], [L], 0, min_bytes=2 * l2, seed=13)
            u, _, _ = time_graph(w, 200, 3, stream)
            pm, _ = time_partition_kernel(w, 50, stream)
            gbs = w.kv_bytes / (u * 1e-6) / 1e9
            if base is None:
                base = u
            rows.append({"workload": name, "page_size": ps, "us_per_step": round(u, 2),
                         "partition_us": round(pm, 2), "kv_gbs": round(gbs, 1),
                         "frac_of_measured_hbm": round(gbs / hbm_peak, 3), "ratio_vs_ps16": round(u / base, 3),
                         "partitions": w.plan().num_partitions, "kernel": kernel_name(w).split(" ")[0]})
            log(f"[bench] small pages {rows[-1]}")
            del w
            torch.cuda.empty_cache()
    return rows


def reduce_max_over_ranks(x: float, device="cpu") -> float:
    """Max of a per-rank float over the process group (identity when not
    distributed): the timed interval of the slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, max_us_per_step: float) -> float:
    """Whole-job throughput: every rank streams its own replica's bytes each
    step; the job's step time is the slowest rank's."""
    return world * bytes_per_rank_step / (max_us_per_step * 1e-6) / 1e9


def kernel_name(wl) -> str:
    p = wl.plan()
    if p.kernel == 2 and wl.ps < 8:
        return f"pa_partition_tc<D={wl.D},{wl.kv},gather> (tcgen05, cp.async page gather)"
    if p.kernel == 2:
        return f"pa_partition_tc<D={wl.D}, {wl.kv}> (tcgen05, TMEM accumulators)"
    if p.kernel == 4:
        return f"pa_partition_u8<N={p.row_tiles}, page {wl.ps}> (tcgen05, keys on M, u8 codes converted into TMEM)"
    if p.kernel == 1:
        return f"pa_partition_f32<D={wl.D}>"
    if wl.ps < 8:
        return f"pa_partition_mma<D={wl.D},{wl.kv},gather> (mma.sync, one bulk copy per key row)"
    return f"pa_partition_mma<D={wl.D}, {wl.kv}, n-tiles={p.row_tiles}> (mma.sync)"


def l2_bytes():
    import torch
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20))


def capture_graph(wl, steps_in_graph, stream):
    """Capture `steps_in_graph` verify steps rotating over the replicas."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for r in range(min(wl.replicas, steps_in_graph)):  # warm every replica eagerly
            wl.forward(r, stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for s in range(steps_in_graph):
                wl.forward(s % wl.replicas, stream)
    return g


def time_graph(wl, steps, warmup, stream, min_seconds=0.0):
    """Median over trials of (device time of `steps` steps) / steps, in µs.
    Each trial replays graphs of a fixed number of steps; trials repeat until
    min_seconds of device time (so a clock sampler sees the load)."""
    import torch
    per_graph = max(1, min(steps, 64))
    n_graphs = max(1, steps // per_graph)
    exact = per_graph * n_graphs
    g = capture_graph(wl, per_graph, stream)
    trials = []
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(max(1, warmup)):
            g.replay()
        torch.cuda.synchronize()
        t_start = time.time()
        while True:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_graphs):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            trials.append(e0.elapsed_time(e1) * 1e3 / exact)
            if time.time() - t_start >= min_seconds and len(trials) >= 3:
                break
    return statistics.median(trials), exact, trials


def time_steps_eager(wl, n, warmup, stream):
    """Per-call device time (µs) of n single verify steps, each between two
    events on the launching stream (replicas rotated so the KV cache exceeds
    L2): the distribution the graph-replayed mean hides."""
    import torch
    out = []
    with torch.cuda.stream(stream):
        for i in range(max(1, warmup)):
            wl.forward(i % wl.replicas, stream)
        torch.cuda.synchronize()
        for i in range(n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            wl.forward(i % wl.replicas, stream)
            e1.record(stream)
            e1.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3)
    return out


def pct(xs, q):
    """q-th percentile (0..100) of xs, nearest rank."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q / 100.0 * (len(ys) - 1)))))]


def time_calls(fn, replicas, stream, reps=64, trials=20):
    """Median device time (µs) of one fn(r) call: a CUDA graph of `reps`
    back-to-back calls rotating r over the replicas, replayed between two
    events on the launching stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for r in range(min(replicas, reps)):
            fn(r)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                fn(r % replicas)
        res = []
        for _ in range(trials):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            res.append(e0.elapsed_time(e1) * 1e3 / reps)
    return statistics.median(res)


def time_partition_kernel(wl, steps, stream):
    """Average device duration of the partition kernel: a CUDA graph of
    `steps` back-to-back partition launches (rotating replicas), replayed
    between two events on the launching stream.  Returns (mean, median) µs
    over trials."""
    import torch
    reps = max(1, min(steps, 64))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for r in range(min(wl.replicas, reps)):
            wl.partition(r % wl.replicas, stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                wl.partition(r % wl.replicas, stream)
        res = []
        for _ in range(max(5, steps // reps)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            res.append(e0.elapsed_time(e1) * 1e3 / reps)
    return statistics.mean(res), statistics.median(res)


def time_e2e(wl, steps, warmup, stream, graph=True):
    """Through the public API with host buffers: every step copies its query
    tokens, block table, past_lens and subsequence_begins from pinned host
    memory, runs the verify step, and copies the output back to pinned host
    memory, all inside the timed region.  The step's inputs are packed in one
    pinned host buffer ([q | block table | past_lens | begins], each part
    16-byte aligned) and move with one host-to-device copy into a device
    buffer the call's input pointers point into; the output comes back with
    one device-to-host copy.  The KV cache is resident device state (the cache
    of a serving engine), as it is between verify steps.  graph=True captures
    the per-step sequence (copies + launches) in a CUDA graph, as a serving
    loop would; graph=False issues it eagerly."""
    import torch
    import paged_attention_speculative_gb300 as pa

    def align16(n):
        return (n + 15) // 16 * 16

    q_bytes = wl.q.numel() * wl.q.element_size()
    bt_bytes = wl.block_tables[0].numel() * 4
    pl_bytes = wl.past_lens.numel() * 4
    sb_bytes = wl.begins.numel() * 4
    o_bt = align16(q_bytes)
    o_pl = o_bt + align16(bt_bytes)
    o_sb = o_pl + align16(pl_bytes)
    total = o_sb + align16(sb_bytes)
    # one packed host buffer per replica (its block table differs)
    host = torch.empty((wl.replicas, total), dtype=torch.uint8).pin_memory()
    for r in range(wl.replicas):
        host[r, :q_bytes] = wl.q.cpu().view(torch.uint8).reshape(-1)
        host[r, o_bt:o_bt + bt_bytes] = wl.block_tables_host[r].view(torch.uint8).reshape(-1)
        host[r, o_pl:o_pl + pl_bytes] = wl.past_lens.cpu().view(torch.uint8).reshape(-1)
        host[r, o_sb:o_sb + sb_bytes] = wl.begins.cpu().view(torch.uint8).reshape(-1)
    dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    q_d = dev[:q_bytes].view(wl.q.dtype).view(wl.q.shape)
    bt_d = dev[o_bt:o_bt + bt_bytes].view(torch.int32).view(wl.block_tables[0].shape)
    pl_d = dev[o_pl:o_pl + pl_bytes].view(torch.int32)
    sb_d = dev[o_sb:o_sb + sb_bytes].view(torch.int32)
    out_h = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()

    def step(s):
        dev.copy_(host[s % wl.replicas], non_blocking=True)
        pa.forward(q_d, wl.k, wl.v, bt_d, pl_d, sb_d, wl.max_ctx, wl.scale, wl.window, wl.kv_code,
                   wl.out, wl.dims, wl.ws, stream=stream)
        out_h.copy_(wl.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(warmup):
            step(s)
        torch.cuda.synchronize()
        if graph:
            reps = max(1, min(steps, 32))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for s in range(reps):
                    step(s)
            g.replay()
            torch.cuda.synchronize()
            n = max(1, steps // reps)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            done = n * reps
        else:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for s in range(steps):
                step(s)
            e1.record(stream)
            e1.synchronize()
            done = steps
    got = out_h.float()
    assert torch.isfinite(got).all(), "end-to-end output not finite"
    us = e0.elapsed_time(e1) * 1e3 / done
    h2d = total
    d2h = wl.out.numel() * wl.out.element_size()
    return us, h2d, d2h


def time_e2e_pipelined(wl, steps, warmup, stream):
    """Like time_e2e (packed host inputs, one H2D and one D2H per step, all
    inside the timed region) with the copies on two copy streams and two
    device input / output buffers, as a serving loop overlaps them: step i's
    host-to-device copy runs while step i-1 computes, and its device-to-host
    copy while step i+1 computes.  Events order each buffer's reuse; the
    per-step sequence is captured in one CUDA graph of 32 steps."""
    import torch
    import paged_attention_speculative_gb300 as pa

    def align16(n):
        return (n + 15) // 16 * 16

    q_bytes = wl.q.numel() * wl.q.element_size()
    bt_bytes = wl.block_tables[0].numel() * 4
    pl_bytes = wl.past_lens.numel() * 4
    sb_bytes = wl.begins.numel() * 4
    o_bt = align16(q_bytes)
    o_pl = o_bt + align16(bt_bytes)
    o_sb = o_pl + align16(pl_bytes)
    total = o_sb + align16(sb_bytes)
    host = torch.empty((wl.replicas, total), dtype=torch.uint8).pin_memory()
    for r in range(wl.replicas):
        host[r, :q_bytes] = wl.q.cpu().view(torch.uint8).reshape(-1)
        host[r, o_bt:o_bt + bt_bytes] = wl.block_tables_host[r].view(torch.uint8).reshape(-1)
        host[r, o_pl:o_pl + pl_bytes] = wl.past_lens.cpu().view(torch.uint8).reshape(-1)
        host[r, o_sb:o_sb + sb_bytes] = wl.begins.cpu().view(torch.uint8).reshape(-1)
    devs = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
    views = []
    for dv in devs:
        views.append((dv[:q_bytes].view(wl.q.dtype).view(wl.q.shape),
                      dv[o_bt:o_bt + bt_bytes].view(torch.int32).view(wl.block_tables[0].shape),
                      dv[o_pl:o_pl + pl_bytes].view(torch.int32), dv[o_sb:o_sb + sb_bytes].view(torch.int32)))
    outs = [torch.empty_like(wl.out) for _ in range(2)]
    outs_h = [torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory() for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def run(first, n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        ev_got = [torch.cuda.Event() for _ in range(n)]
        h2d_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev_out[i - 2])  # the step that read this input buffer is done
                devs[k].copy_(host[(first + i) % wl.replicas], non_blocking=True)
                ev_in[i].record(h2d_s)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_got[i - 2])  # this output buffer has been read back
            q_d, bt_d, pl_d, sb_d = views[k]
            pa.forward(q_d, wl.k, wl.v, bt_d, pl_d, sb_d, wl.max_ctx, wl.scale, wl.window, wl.kv_code,
                       outs[k], wl.dims, wl.ws, stream=stream)
            ev_out[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_out[i])
                outs_h[k].copy_(outs[k], non_blocking=True)
                ev_got[i].record(d2h_s)
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)

    with torch.cuda.stream(stream):
        run(0, max(2, warmup))
        torch.cuda.synchronize()
        reps = 32
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(0, reps)
        g.replay()
        torch.cuda.synchronize()
        n = max(1, steps // reps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        e1.synchronize()
    for oh in outs_h:
        assert torch.isfinite(oh.float()).all(), "end-to-end output not finite"
    us = e0.elapsed_time(e1) * 1e3 / (n * reps)
    return us, total, wl.out.numel() * wl.out.element_size()


# ---------------------------------------------------------------------------
# Clocks during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[0] == "0":
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        loaded = [s for s in sm if s is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, nm in enumerate(names):
            if any(r[5 + i].lower() == "active" for r in rows):
                reasons.append(nm)
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------
# Oracle (CPU fp64) timing: a bounded sample of the same workload.
# ---------------------------------------------------------------------------
def oracle_sample_step(T, L, seed=0):
    """One KV head's GQA group (all T tokens x 4 query heads) of the headline
    workload, over all L+T keys: 1/8 of a step's rows and KV bytes."""
    import numpy as np
    from paged_attention_speculative_gb300 import workloads as W
    case = W.make_case("oracle_sample", seed=seed, query_lens=[T], past_lens=[L], num_q_heads=4, num_kv_heads=1,
                       head_dim=128, page_size=16, poison=False, extra_block_frac=0.01)
    kv_bytes = (L + T) * 1 * 2 * 128 * 2
    return case, kv_bytes


def time_oracle(T, L, min_seconds, steps=None):
    import oracle
    oracle.build()
    case, kv_bytes = oracle_sample_step(T, L)
    cores = oracle.max_threads()

    def one():
        oracle.forward(case.q, case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                       case.past_lens, case.subsequence_begins, num_q_heads=4, num_kv_heads=1, head_dim=128,
                       page_size=16, num_blocks=case.num_blocks, scale=case.scale)
    one()  # warm
    n = 0
    t0 = time.perf_counter()
    while True:
        one()
        n += 1
        el = time.perf_counter() - t0
        if steps is not None and n >= steps:
            break
        if steps is None and el >= min_seconds and n >= 2:
            break
    per = el / n
    return kv_bytes / per / 1e9, per, n, cores


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_attention_speculative_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(config_name):
    """DRAM bytes per partition launch from the committed ncu summary, only if
    it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("per_launch_bytes", {}).get(config_name)


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    T, L = HEADLINE["q_lens"][0], HEADLINE["past"][0]
    for _ in range(args.warmup):
        pass
    gbs, per, n, cores = time_oracle(T, L, 0, steps=args.steps)
    line = {"impl": "reference", "metric": "KV-read GB/s per verify step (T=4, L=32768, Qwen-like GQA)",
            "value": gbs, "unit": "GB/s", "n_gpus": args.gpus, "steps": n, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE["name"] + " (oracle sample: one KV head's 4x4 query rows)",
                       "global_batch": 1, "seq_len": L + T, "parallelism": "cpu"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: all 4 new tokens x the 4 query heads of one KV head over all "
                                       f"{L + T} keys (1/8 of the step's rows and KV bytes)",
                             "cpu": cpu_model()},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world):
    import torch
    import paged_attention_speculative_gb300 as pa
    from paged_attention_speculative_gb300 import build as _build
    dist = None
    if world > 1:
        import torch.distributed as dist
    if rank == 0 or world == 1:
        _build.build()
    if dist is not None:
        dist.barrier()
    pa.load_library()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    stream = torch.cuda.Stream()
    L2 = l2_bytes()
    pk = peaks()
    hbm_peak = pk.get("hbm_gbs")
    peak_kind = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0

    H = HEADLINE
    wl = DeviceWorkload(H["Hq"], H["Hkv"], H["D"], H["ps"], H["kv"], H["q_lens"], H["past"], H["window"],
                        min_bytes=2 * L2, seed=rank)
    log(f"[bench] headline {H['name']}: replicas={wl.replicas} plan={wl.plan().as_dict()}")

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    us, exact, trials = time_graph(wl, args.steps, args.warmup, stream, min_seconds=args.min_seconds)
    clk = clocks.stop()
    torch.cuda.synchronize()
    if dist is not None:
        us = reduce_max_over_ranks(us, device="cuda")
        dist.barrier()
    value = whole_job_gbs(wl.kv_bytes, world, us)

    eager = time_steps_eager(wl, 60, 10, stream)
    part_mean, part_med = time_partition_kernel(wl, max(args.steps, 20), stream)
    achieved = wl.kv_bytes / (part_mean * 1e-6) / 1e9
    e2e_us, h2d, d2h = time_e2e_pipelined(wl, max(args.steps, 64), args.warmup, stream)
    e2e_seq_us, _, _ = time_e2e(wl, max(args.steps, 20), args.warmup, stream, graph=True)
    e2e_eager_us, _, _ = time_e2e(wl, max(args.steps, 20), args.warmup, stream, graph=False)
    e2e_value = world * wl.kv_bytes / (e2e_us * 1e-6) / 1e9

    # T=1 at the same context (the ratio the pages' fix is about)
    wl1 = DeviceWorkload(H["Hq"], H["Hkv"], H["D"], H["ps"], H["kv"], [1], H["past"], H["window"],
                         min_bytes=2 * L2, seed=rank + 7)
    us1, _, _ = time_graph(wl1, args.steps, args.warmup, stream)
    del wl1

    sweep = []
    if not args.no_sweep and rank == 0:
        for fam in SWEEP:
            for L in fam["L"]:
                base = None
                for T in fam["T"]:
                    w = DeviceWorkload(fam["Hq"], fam["Hkv"], fam["D"], fam["ps"], fam["kv"], [T], [L], fam["window"],
                                       min_bytes=2 * L2, seed=3)
                    u, _, _ = time_graph(w, 200, 3, stream)
                    pm, _ = time_partition_kernel(w, 50, stream)
                    gbs = w.kv_bytes / (u * 1e-6) / 1e9
                    if base is None:
                        base = u
                    sweep.append({"workload": fam["name"].format(T=T, L=L), "us_per_step": round(u, 2),
                                  "partition_us": round(pm, 2), "kv_mb": round(w.kv_bytes / 1e6, 2),
                                  "kv_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 3),
                                  "ratio_vs_T1": round(u / base, 3), "tflops": round(w.flops / (u * 1e-6) / 1e12, 1),
                                  "partitions": w.plan().num_partitions, "kernel": kernel_name(w).split(" ")[0]})
                    log(f"[bench] {sweep[-1]}")
                    del w
                    torch.cuda.empty_cache()
        # batched mix (a): batch 8, T ~ U{1..4}, past ~ U[2000, 4000], window 1024
        import random
        rr = random.Random(1000)
        Ts = [rr.randint(1, 4) for _ in range(8)]
        Ls = [rr.randint(2000, 4000) for _ in range(8)]
        for tag, qs in (("mix_a", Ts), ("mix_a_all_T1", [1] * 8)):
            w = DeviceWorkload(32, 16, 256, 64, "bf16", qs, Ls, 1024, min_bytes=2 * L2, seed=5)
            u, _, _ = time_graph(w, 200, 3, stream)
            gbs = w.kv_bytes / (u * 1e-6) / 1e9
            sweep.append({"workload": tag, "us_per_step": round(u, 2), "kv_mb": round(w.kv_bytes / 1e6, 2),
                          "kv_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 3),
                          "partitions": w.plan().num_partitions})
            log(f"[bench] {sweep[-1]}")
            del w
        mix = [s for s in sweep if s["workload"].startswith("mix_a")]
        if len(mix) == 2:
            mix[0]["ratio_vs_T1"] = round(mix[0]["us_per_step"] / mix[1]["us_per_step"], 3)

    # The cache update (the step before the verify: the new tokens' K/V into
    # their pages) alone, and followed by the verify step.
    cache_update = []
    if not args.no_sweep and rank == 0:
        cfgs = [("qwen_gqa_T4_L32768", 32, 8, 128, 16, "bf16", [4], [32768]),
                ("qwen_u8_T3_L32768", 32, 8, 128, 16, "u8", [3], [32768]),
                ("batch64_T4_L4096_bf16", 32, 8, 128, 16, "bf16", [4] * 64, [4096] * 64),
                ("batch64_T4_L4096_u8", 32, 8, 128, 16, "u8", [4] * 64, [4096] * 64)]
        for name, hq, hkv, d, ps, kvd, qs, ls in cfgs:
            w = DeviceWorkload(hq, hkv, d, ps, kvd, qs, ls, 0, min_bytes=2 * L2, seed=9)
            u_upd = time_calls(lambda r: w.cache_update(r, stream), w.replicas, stream)
            u_step = time_calls(lambda r: (w.cache_update(r, stream), w.forward(r, stream)), w.replicas, stream)
            u_fwd = time_calls(lambda r: w.forward(r, stream), w.replicas, stream)
            cache_update.append({"workload": name, "update_us": round(u_upd, 2), "update_bytes": w.update_bytes,
                                 "update_gbs": round(w.update_bytes / (u_upd * 1e-6) / 1e9, 1),
                                 "update_frac_of_measured_hbm": round(w.update_bytes / (u_upd * 1e-6) / 1e9 / hbm_peak, 4),
                                 "update_then_verify_us": round(u_step, 2), "verify_us": round(u_fwd, 2)})
            log(f"[bench] cache update {cache_update[-1]}")
            del w
            torch.cuda.empty_cache()

    # Tree-mask verify: a random 8-node draft tree per sequence against the
    # causal chain of 8 tokens on the same cache.
    tree_verify = []
    if not args.no_sweep and rank == 0:
        import random
        for name, hq, hkv, d, ps, kvd, T, L in (("qwen_gqa_T8_L32768", 32, 8, 128, 16, "bf16", 8, 32768),
                                                  ("long_T8_L131072", 64, 8, 128, 16, "bf16", 8, 131072),
                                                  ("qwen_u8_T8_L32768", 32, 8, 128, 16, "u8", 8, 32768)):
            w = DeviceWorkload(hq, hkv, d, ps, kvd, [T], [L], 0, min_bytes=2 * L2, seed=11)
            rr = random.Random(7)
            m = []
            for i in range(T):
                parent = -1 if i == 0 else rr.randint(-1, i - 1)
                m.append((1 << i) | (m[parent] if parent >= 0 else 0))
            tm = torch.tensor(m, dtype=torch.uint8, device="cuda")
            u_tree = time_calls(lambda r: w.forward_tree(r, tm, stream), w.replicas, stream)
            u_chain = time_calls(lambda r: w.forward(r, stream), w.replicas, stream)
            tree_verify.append({"workload": name, "tree_masks": m, "tree_us": round(u_tree, 2),
                                "chain_us": round(u_chain, 2), "ratio": round(u_tree / u_chain, 3),
                                "kv_gbs_tree": round(w.kv_bytes / (u_tree * 1e-6) / 1e9, 1)})
            log(f"[bench] tree verify {tree_verify[-1]}")
            del w
            torch.cuda.empty_cache()

    small_pages = small_page_sweep(stream, hbm_peak, L2) if (not args.no_sweep and rank == 0) else []
    mixed = mixed_sweep(stream, hbm_peak, L2) if (not args.no_sweep and rank == 0) else []

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, per, n, cores = time_oracle(H["q_lens"][0], H["past"][0], args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} oracle steps, each all 4 new tokens x the 4 query heads of one KV head over all "
                         f"{H['past'][0] + 4} keys (1/8 of the headline step), {per:.3f} s each",
               "cpu": cpu_model()}

    if rank != 0:
        return
    line = {
        "metric": "KV-read GB/s per verify step (T=4, L=32768, Qwen-like GQA)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": exact, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "us_per_step": us, "us_per_step_T1": us1, "ratio_vs_T1": us / us1,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": H["name"], "global_batch": world, "seq_len": H["past"][0] + H["q_lens"][0],
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "heads": "32q/8kv", "head_dim": 128, "page_size": 16, "kv_dtype": "bf16",
                   "l2": f"KV cache rotated over {wl.replicas} replicas ({wl.replicas * wl.total_device_bytes / 2**20:.0f}"
                         f" MiB > 2x L2)", "launch": "CUDA graph replay", "trials": len(trials)},
        "us_per_step_trials": {"p10": pct(trials, 10), "p50": pct(trials, 50), "p90": pct(trials, 90),
                               "n": len(trials), "what": f"graph replay, each trial the mean of {exact} steps"},
        "us_per_call_eager": {"p10": pct(eager, 10), "p50": pct(eager, 50), "p90": pct(eager, 90), "n": len(eager),
                              "what": "one pa_verify_forward call between two events, 10 warm-up calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": measured_traffic(H["name"]),
                     "frac_of_nominal_8tbs": achieved / 8000.0,
                     "kernel": kernel_name(wl),
                     "kernel_us_mean": part_mean, "kernel_timing": "CUDA graph of back-to-back partition launches",
                     "kernel_us_median": part_med, "algorithmic_bytes_per_launch": wl.kv_bytes,
                     "peak_kind": f"{peak_kind} copy rate (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": e2e_us,
                "launch": "CUDA graph of 32 steps, each one packed H2D copy + forward + one D2H copy; copies on "
                          "two copy streams overlap the neighbouring steps' kernels (double-buffered inputs and outputs)",
                "sequential_us_per_step": e2e_seq_us,
                "eager_us_per_step": e2e_eager_us,
                "eager_value": world * wl.kv_bytes / (e2e_eager_us * 1e-6) / 1e9},
        "cpu_baseline": cpu,
        "clocks": clk,
        "gpu_launches": exact * wl.launches_per_step(),
        "sweep": sweep,
        "cache_update": cache_update,
        "tree_verify": tree_verify,
        "small_pages": small_pages,
        "mixed": mixed,
    }
    print(json.dumps(line), flush=True)


# Workloads the ncu summaries of the other kernels are taken on: the
# page gathers (one token per page), a prefill chunk alone, and others.
PROFILE_EXTRA = {
    "long_T8_L131072_ps1": dict(Hq=64, Hkv=8, D=128, ps=1, kv="bf16", q_lens=[8], past=[131072], window=0),
    # head_dim 256 in one-token pages: the warp-level kernel's per-key bulk copies
    "gemma_global_T2_L32768_ps1": dict(Hq=32, Hkv=16, D=256, ps=1, kv="bf16", q_lens=[2], past=[32768], window=0),
    # u8 with 64 query rows per KV head: the warp-level kernel's u8 path
    "long_u8_T8_L32768": dict(Hq=64, Hkv=8, D=128, ps=16, kv="u8", q_lens=[8], past=[32768], window=0),
    # the cache update before each verify step (64 sequences of 4 new tokens)
    "update_batch64_T4_L4096": dict(Hq=32, Hkv=8, D=128, ps=16, kv="bf16", q_lens=[4] * 64, past=[4096] * 64,
                                    window=0, update=True),
    "prefill_T512_L32768": dict(Hq=32, Hkv=8, D=128, ps=16, kv="bf16", q_lens=[512], past=[32768], window=0,
                                mixed=True),
    # a short chunk at long context: its blocks' keys split into pieces
    "prefill_T64_L32768": dict(Hq=32, Hkv=8, D=128, ps=16, kv="bf16", q_lens=[64], past=[32768], window=0,
                               mixed=True),
}


def workload_by_name(name):
    """A sweep / headline workload spec by its printed name, e.g. qwen_gqa_T4_L32768."""
    if name == HEADLINE["name"]:
        return dict(HEADLINE)
    if name in PROFILE_EXTRA:
        return dict(name=name, **PROFILE_EXTRA[name])
    for fam in SWEEP:
        for L in fam["L"]:
            for T in fam["T"]:
                if fam["name"].format(T=T, L=L) == name:
                    return dict(name=name, Hq=fam["Hq"], Hkv=fam["Hkv"], D=fam["D"], ps=fam["ps"], kv=fam["kv"],
                                q_lens=[T], past=[L], window=fam["window"])
    raise SystemExit(f"unknown workload {name}")


def run_profile(args):
    """Eager verify steps of one workload and nothing else: the command the
    ncu summaries under profiles/ were taken with."""
    import torch
    import paged_attention_speculative_gb300 as pa
    from paged_attention_speculative_gb300 import build as _build
    _build.build()
    pa.load_library()
    spec = workload_by_name(args.profile)
    wl = DeviceWorkload(spec["Hq"], spec["Hkv"], spec["D"], spec["ps"], spec["kv"], spec["q_lens"], spec["past"],
                        spec["window"], min_bytes=2 * l2_bytes())
    stream = torch.cuda.Stream()
    step = wl.forward_mixed if spec.get("mixed") else wl.forward
    with torch.cuda.stream(stream):
        for s in range(args.warmup + args.steps):
            if spec.get("update"):
                wl.cache_update(s % wl.replicas, stream)
            step(s % wl.replicas, stream)
    torch.cuda.synchronize()
    log(f"[profile] {spec['name']}: {args.warmup + args.steps} steps, plan {wl.plan().as_dict()}, "
        f"kv bytes/step {wl.kv_bytes}")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-seconds", type=float, default=2.0, help="keep the timed loop busy this long (clocks)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", default=None, help="run eager steps of one named workload only (for ncu)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile:
        run_profile(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
