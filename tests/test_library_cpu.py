"""Host-side checks that need no GPU: the library builds and loads, exports
every entry point include/pa_verify.h declares, the partition heuristic's
properties, and host-detected argument errors (which return before any CUDA
call)."""
import ctypes
import math
import os
import re

import pytest

import paged_attention_speculative_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_attention_speculative_gb300 import build
    build.build()
    return pa.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa_verify.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_(?:verify|cache|mixed|forward)_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"libpa_verify.so does not export {n}"
    assert set(names) == set(pa.EXPORTED)


def dims(**kw):
    base = dict(num_seqs=1, total_tokens=4, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                num_blocks=3000, max_blocks_per_seq=2100, q_dtype=pa.PA_BF16, out_dtype=pa.PA_BF16)
    base.update(kw)
    return pa.PaDims(**base)


def test_plan_fills_the_sms_once_at_long_context(lib):
    # head_dim 64, 4 rows per KV head: the warp-level kernel, two CTAs per SM
    p = pa.plan(dims(total_tokens=1, head_dim=64), 32769, 0, pa.PA_BF16, 152)
    assert p.kernel == 0 and p.row_tiles == 1
    assert p.part_tokens % max(p.stage_keys, 16) == 0
    assert p.num_partitions * p.part_tokens >= 32769
    assert (p.num_partitions - 1) * p.part_tokens < 32769
    assert 0.8 * 304 <= p.ctas <= 1.1 * 304
    # 16 rows per KV head: the tensor-memory kernel, one CTA per SM
    t = pa.plan(dims(), 32772, 0, pa.PA_BF16, 152)
    assert t.kernel == 2 and t.stage_keys == 64
    assert 0.8 * 152 <= t.ctas <= 1.1 * 152


def test_plan_u8_partitions_on_page_quantum(lib):
    # the u8 tensor-memory kernel's partitions are whole pages, not whole
    # 128-key stages: 32771 keys over 152 CTAs -> 1728 keys each (13.5 stages)
    u = pa.plan(dims(total_tokens=3), 32771, 0, pa.PA_U8, 152)
    assert u.kernel == 4 and u.stage_keys == 128
    assert u.part_tokens == 1728 and u.num_partitions == 19
    u64 = pa.plan(dims(total_tokens=1, page_size=64), 65536, 0, pa.PA_U8, 152)
    assert u64.kernel == 4 and u64.part_tokens % 64 == 0
    assert (u64.num_partitions - 1) * u64.part_tokens < 65536 <= u64.num_partitions * u64.part_tokens


def test_plan_independent_of_query_count(lib):
    """The split must not collapse when a sequence brings more than one
    query token (the failure both OpenVINO issue 38153 and the
    dual-radeon-vllm article describe)."""
    ps = [pa.plan(dims(total_tokens=t), 32768 + t, 0, pa.PA_BF16, 152).num_partitions for t in (2, 3, 4)]
    assert min(ps) == max(ps) and ps[0] > 16
    # T=1 (4 rows) keeps the split too
    assert pa.plan(dims(total_tokens=1), 32769, 0, pa.PA_BF16, 152).num_partitions >= ps[0]
    # and on the warp-level kernel (head_dim 64, two CTAs per SM) T = 1..4 split alike
    ps64 = [pa.plan(dims(total_tokens=t, head_dim=64), 32768 + t, 0, pa.PA_BF16, 152).num_partitions
            for t in (1, 2, 3, 4)]
    assert min(ps64) >= 16


def test_plan_window_reads_only_the_window(lib):
    d = dims(num_kv_heads=16, head_dim=256, page_size=64, total_tokens=2)
    full = pa.plan(d, 32770, 0, pa.PA_BF16, 152)
    swa = pa.plan(d, 32770, 1024, pa.PA_BF16, 152)
    assert swa.num_partitions * swa.part_tokens >= 1024 + 1
    assert swa.num_partitions * swa.part_tokens <= 1024 + 2 + 2 * 64 + swa.part_tokens
    assert full.num_partitions * full.part_tokens >= 32770


def test_plan_bounds_partial_traffic(lib):
    """Per-token partials (rows x (D+2) x 4 bytes per partition) stay near
    10 % of the KV bytes a partition streams."""
    for t, g, hkv, d in [(8, 8, 8, 128), (4, 4, 8, 128), (2, 2, 16, 256)]:
        dd = dims(total_tokens=t, num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=d)
        p = pa.plan(dd, 8192 + t, 0, pa.PA_BF16, 152)
        partial = t * g * (d + 2) * 4
        kv = p.part_tokens * 2 * d * 2
        assert partial <= 0.11 * kv


def test_plan_scales_with_sm_count(lib):
    d = dims(max_blocks_per_seq=8200)
    a = pa.plan(d, 131072, 0, pa.PA_BF16, 76)
    b = pa.plan(d, 131072, 0, pa.PA_BF16, 152)
    assert b.num_partitions > a.num_partitions


def test_plan_rejections(lib):
    p = pa.PaPlan()
    cases = [
        (dims(head_dim=96), pa.PA_BF16, -4),
        (dims(head_dim=64), pa.PA_U8, -4),
        (dims(page_size=12), pa.PA_BF16, -5),
        (dims(page_size=3), pa.PA_BF16, -5),
        (dims(page_size=512), pa.PA_BF16, -5),
        (dims(page_size=4), pa.PA_U8, -5),
        (dims(page_size=2, head_dim=256, num_q_heads=64, total_tokens=8), pa.PA_BF16, -10),  # 64 rows > 32
        (dims(page_size=1, head_dim=256), pa.PA_U8, -5),
        (dims(page_size=1, num_q_heads=128, num_kv_heads=8, total_tokens=8, max_blocks_per_seq=8192), pa.PA_BF16,
         -5),
        (dims(num_q_heads=30), pa.PA_BF16, -3),
        (dims(q_dtype=pa.PA_F16), pa.PA_BF16, -2),
        (dims(out_dtype=pa.PA_U8), pa.PA_BF16, -2),
        (dims(num_q_heads=128, num_kv_heads=8, total_tokens=8), pa.PA_BF16, -10),
    ]
    for d, kv, want in cases:
        assert lib.pa_verify_plan(ctypes.byref(d), 4096, 0, kv, 152, ctypes.byref(p)) == want
    assert lib.pa_verify_plan(ctypes.byref(dims()), 0, 0, pa.PA_BF16, 152, ctypes.byref(p)) == -8
    assert lib.pa_verify_plan(ctypes.byref(dims()), 2100 * 16 + 1, 0, pa.PA_BF16, 152, ctypes.byref(p)) == -8
    assert lib.pa_verify_plan(None, 4096, 0, pa.PA_BF16, 152, ctypes.byref(p)) == -1


def test_plan_small_pages(lib):
    """Pages of 1, 2 or 4 tokens: 16-bit caches take the tensor-memory kernel
    (its cp.async-gather producer) whatever the row count, with partitions
    free of the per-CTA page-list cap; head_dim 256 takes the warp-level
    kernel with per-key bulk copies (two CTAs per SM, the same partitions as
    8-token pages); fp32 caches keep the FFMA kernel."""
    p = pa.PaPlan()
    for ps in (1, 2, 4):
        for hq, t in ((32, 1), (32, 4), (64, 8)):
            d = dims(page_size=ps, num_q_heads=hq, total_tokens=t, max_blocks_per_seq=131072 // ps + 8)
            assert lib.pa_verify_plan(ctypes.byref(d), 131072 + t, 0, pa.PA_BF16, 152, ctypes.byref(p)) == 0
            assert p.kernel == 2 and p.part_tokens % 64 == 0
            assert p.part_tokens > 1024  # more pages per CTA than a staged page list holds
            assert p.num_partitions * p.part_tokens >= 131072 + t
        d = dims(page_size=ps, head_dim=64, num_q_heads=8, num_kv_heads=2, total_tokens=3, q_dtype=pa.PA_F16)
        assert lib.pa_verify_plan(ctypes.byref(d), 600, 0, pa.PA_F16, 152, ctypes.byref(p)) == 0
        assert p.kernel == 2
        d = dims(page_size=ps, q_dtype=pa.PA_F32, max_blocks_per_seq=4096)
        assert lib.pa_verify_plan(ctypes.byref(d), 4000, 0, pa.PA_F32, 152, ctypes.byref(p)) == 0
        assert p.kernel == 1
        for hq, t, window in ((32, 2, 0), (32, 8, 0), (64, 4, 0), (32, 2, 1024)):
            d = dims(page_size=ps, head_dim=256, num_q_heads=hq, num_kv_heads=16, total_tokens=t,
                     max_blocks_per_seq=32768 // ps + 8)
            assert lib.pa_verify_plan(ctypes.byref(d), 32768 + t, window, pa.PA_BF16, 152, ctypes.byref(p)) == 0
            assert p.kernel == 0 and p.stage_keys == 32 and p.row_tiles == 1
            assert 2 * (p.smem_bytes + 1024) <= 233472  # two CTAs per SM
            assert p.num_partitions * p.part_tokens >= (window + t - 1 if window else 32768 + t)
            d8 = dims(page_size=8, head_dim=256, num_q_heads=hq, num_kv_heads=16, total_tokens=t,
                      max_blocks_per_seq=32768 // 8 + 8)
            q = pa.PaPlan()
            assert lib.pa_verify_plan(ctypes.byref(d8), 32768 + t, window, pa.PA_BF16, 152, ctypes.byref(q)) == 0
            assert (q.kernel, q.num_partitions, q.part_tokens) == (0, p.num_partitions, p.part_tokens)


def test_forward_host_errors_need_no_gpu(lib):
    d = dims()
    z = ctypes.c_void_p(0)
    a16 = ctypes.c_void_p(4096)
    args = [a16, a16, a16, a16, a16, a16, 4096, 0.1, 0, pa.PA_BF16, a16, ctypes.byref(d), a16, 1 << 20, z]
    bad = list(args)
    bad[0] = z
    assert lib.pa_verify_forward(*bad) == -1
    bad = list(args)
    bad[0] = ctypes.c_void_p(4098)
    assert lib.pa_verify_forward(*bad) == -6
    bad = list(args)
    bad[9] = pa.PA_F16
    assert lib.pa_verify_forward(*bad) == -2
    bad = list(args)
    bad[11] = None
    assert lib.pa_verify_forward(*bad) == -1


def test_no_alloc_rejections_come_before_any_cuda_call(lib):
    """pa_verify_forward_no_alloc checks its arguments before it resolves its
    scratch or enqueues anything: on a machine without a GPU, where any CUDA
    call fails (PA_ERR_CUDA), a bad argument still returns its own code."""
    a16 = ctypes.c_void_p(4096)
    z = ctypes.c_void_p(0)

    def call(d, kv=pa.PA_BF16, q=a16, out=a16, mcl=4096):
        return lib.pa_verify_forward_no_alloc(q, a16, a16, a16, a16, a16, mcl, 0.1, 0, kv, out, ctypes.byref(d), z)
    assert call(dims(head_dim=96)) == -4
    assert call(dims(q_dtype=pa.PA_F16)) == -2
    assert call(dims(), q=z) == -1
    assert call(dims(), out=ctypes.c_void_p(4100)) == -6
    assert call(dims(), mcl=0) == -8
    assert lib.pa_verify_forward_no_alloc(a16, a16, a16, a16, a16, a16, 4096, 0.1, 0, pa.PA_BF16, a16, None, z) == -1
    # an empty batch is accepted without touching the device
    assert call(dims(total_tokens=0)) == 0


def test_mixed_host_errors_need_no_gpu(lib):
    """pa_forward_mixed rejects what its prefill kernels do not serve before
    touching the device: u8 caches, head_dim 256 with 16-bit caches, 16-bit
    caches with pages under 8 tokens; NULL pointers as pa_verify_forward."""
    a16 = ctypes.c_void_p(4096)
    z = ctypes.c_void_p(0)

    def call(d, kv, ptr=a16):
        return lib.pa_forward_mixed(ptr, a16, a16, a16, a16, a16, 4096, 0.1, 0, kv, a16, ctypes.byref(d), a16,
                                    1 << 20, z)
    assert call(dims(q_dtype=pa.PA_BF16), pa.PA_U8) == -10
    assert call(dims(head_dim=256, num_q_heads=16), pa.PA_BF16) == -10
    assert call(dims(page_size=4, max_blocks_per_seq=4096), pa.PA_BF16) == -5
    assert call(dims(), pa.PA_BF16, ptr=z) == -1


def test_status_strings(lib):
    for code in range(0, -11, -1):
        s = pa.status_string(code)
        assert s and s != "unknown status code"
    assert pa.status_string(-99) == "unknown status code"
