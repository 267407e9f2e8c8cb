"""The cache update on the GPU (pa_cache_update, through the C ABI) against
the oracle's definition: whole caches compared byte for byte (float caches:
values rounded half-even; u8 caches: codes, fp16 scales and zero-points, all
integer decisions taken in binary32 on both sides), then update + verify end
to end against the oracle's update + attention."""
import dataclasses

import numpy as np
import pytest

import oracle
import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import TOL, derived_tolerance, dims, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # name, case factory, new-token dtype
    ("bf16_pages", lambda: W.qwen_gqa(3, 2000, seed=90), "bf16"),
    ("u8_batch", lambda: W.make_case("u8_batch", seed=91, query_lens=[4, 0, 2, 1], past_lens=[14, 3, 31, 0],
                                     num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, kv_dtype="u8"),
     "bf16"),
    ("f16_d64_from_f32", lambda: W.make_case("f16_d64", seed=92, query_lens=[5], past_lens=[61], num_q_heads=8,
                                             num_kv_heads=2, head_dim=64, page_size=8, q_dtype="f16",
                                             kv_dtype="f16"), "f32"),
    ("u8_d256_ps64_from_f16", lambda: W.make_case("u8_d256", seed=93, query_lens=[3, 2], past_lens=[62, 700],
                                                  num_q_heads=32, num_kv_heads=16, head_dim=256, page_size=64,
                                                  kv_dtype="u8", q_dtype="f16"), "f16"),
    ("u8_from_f32_specials", lambda: W.make_case("u8_specials", seed=94, query_lens=[8], past_lens=[100],
                                                 num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=16,
                                                 kv_dtype="u8"), "f32"),
]


def _torch_src(raw, src_dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(raw))
    if src_dtype in ("f16", "bf16"):
        t = t.view(torch.int16).view(torch.float16 if src_dtype == "f16" else torch.bfloat16)
    return t.cuda()


def _gpu_update(case, dev, kn, vn, src_dtype, status=None):
    import torch
    d = dims(case, dev)
    pa.cache_update(_torch_src(kn, src_dtype), _torch_src(vn, src_dtype), dev["k"], dev["v"], dev["bt"], dev["pl"],
                    dev["sb"], d, status=status)
    torch.cuda.synchronize()


def _raw(t):
    import torch
    x = t.cpu()
    if x.dtype in (torch.float16, torch.bfloat16):
        x = x.view(torch.int16)
    return x.numpy().view(np.uint8)


@pytest.mark.parametrize("name,make,src", CASES, ids=[c[0] for c in CASES])
def test_cache_update_matches_the_definition_byte_for_byte(name, make, src):
    case = make()
    kn, vn = W.new_tokens(case, src, seed=3, specials=(name == "u8_from_f32_specials"))
    want_k, want_v = oracle.cache_update(kn, vn, src, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                                         case.past_lens, case.subsequence_begins, num_kv_heads=case.num_kv_heads,
                                         head_dim=case.head_dim, page_size=case.page_size,
                                         num_blocks=case.num_blocks)
    dev = to_device(case)
    _gpu_update(case, dev, kn, vn, src)
    assert np.array_equal(_raw(dev["k"]), np.ascontiguousarray(want_k).view(np.uint8))
    assert np.array_equal(_raw(dev["v"]), np.ascontiguousarray(want_v).view(np.uint8))


@pytest.mark.parametrize("name,make,src", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_update_then_verify_matches_the_oracle(name, make, src):
    import torch
    case = make()
    kn, vn = W.new_tokens(case, src, seed=4)
    kc, vc = oracle.cache_update(kn, vn, src, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                                 case.past_lens, case.subsequence_begins, num_kv_heads=case.num_kv_heads,
                                 head_dim=case.head_dim, page_size=case.page_size, num_blocks=case.num_blocks)
    want = oracle.forward(
        case.q, case.q_dtype, kc, vc, case.kv_dtype, case.block_tables, case.past_lens, case.subsequence_begins,
        num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
        page_size=case.page_size, num_blocks=case.num_blocks, scale=case.scale, sliding_window=case.sliding_window)
    dev = to_device(case)
    _gpu_update(case, dev, kn, vn, src)
    d = dims(case, dev)
    mcl = case.max_context_len
    kvc = {"f32": pa.PA_F32, "f16": pa.PA_F16, "bf16": pa.PA_BF16, "u8": pa.PA_U8}[case.kv_dtype]
    ws = pa.alloc_workspace(d, mcl, case.sliding_window, kvc)
    pa.forward(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], mcl, case.scale, case.sliding_window,
               kvc, dev["out"], d, ws)
    torch.cuda.synchronize()
    got = dev["out"].float().cpu().numpy().astype(np.float64)
    if name == "u8_batch":
        # short contexts (3..35 keys): O(1) outputs, where one rounding of the
        # weights or of the bf16 output alone can exceed 2e-3; use the bound
        # derived from the arithmetic (pa_testing.derived_tolerance) on the
        # updated cache
        upd = dataclasses.replace(case, k_cache=kc, v_cache=vc)
        assert float(np.max(np.abs(got - want) - derived_tolerance(upd, want))) <= 0.0
    else:
        assert float(np.max(np.abs(got - want))) <= TOL


def test_bad_block_id_sets_status_and_skips_the_slot():
    import torch
    case = W.make_case("cu_bad", seed=95, query_lens=[2], past_lens=[15], num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16, kv_dtype="u8")
    kn, vn = W.new_tokens(case, "bf16", seed=5)
    dev = to_device(case)
    before_k = _raw(dev["k"]).reshape(-1).copy()
    # position 15 is valid, position 16 (page 1) points outside the cache
    dev["bt"][0, 1] = case.num_blocks + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _gpu_update(case, dev, kn, vn, "bf16", status=status)
    assert int(status.item()) == 0x4  # PA_STATUS_BLOCK_ID only
    after_k = _raw(dev["k"]).reshape(-1)
    # token 0 (position 15) was written, nothing else changed
    rec = case.page_size * (case.head_dim + 4)
    changed = np.nonzero(after_k != before_k)[0]
    blk0 = int(case.block_tables[0, 0])
    assert changed.size > 0
    assert np.all((changed >= blk0 * case.num_kv_heads * rec) & (changed < (blk0 + 1) * case.num_kv_heads * rec))
