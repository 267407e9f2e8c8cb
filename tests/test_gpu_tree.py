"""Tree-mask verify on the GPU (pa_verify_forward_tree, through the C ABI)
against the oracle's tree definition: random draft trees per sequence on
each default kernel (warp-level mma for head_dim 64 below 8 query rows per
KV head, head_dim 256 and u8; the tensor-memory kernels otherwise; the fp32
path), with windows, batches, empty sequences and one- or many-partition
contexts; and a chain mask must reproduce pa_verify_forward bit for bit."""
import numpy as np
import pytest

import oracle
import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import KV_CODE, TOL, derived_tolerance, dims, run_gpu, to_device

pytestmark = pytest.mark.gpu


def random_tree_masks(case, seed):
    rng = np.random.default_rng(seed)
    m = np.zeros(case.total_tokens, dtype=np.uint8)
    for b in range(case.num_seqs):
        t0 = int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            parent = -1 if i == 0 else int(rng.integers(-1, i))
            m[t0 + i] = (1 << i) | (m[t0 + parent] if parent >= 0 else 0)
    return m


CASES = [
    # (case, kernel the plan picks, short context -> derived bound)
    (lambda: W.make_case("tree_mma", seed=101, query_lens=[7], past_lens=[3000], num_q_heads=8, num_kv_heads=8,
                         head_dim=64, page_size=16), 0, False),
    (lambda: W.qwen_gqa(8, 2500, seed=102), 2, False),
    (lambda: W.long_ctx_b(3000, seed=103), 2, False),
    (lambda: W.make_case("tree_batch_win", seed=104, query_lens=[5, 0, 8, 3], past_lens=[900, 10, 1300, 40],
                         num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, sliding_window=400), 2, True),
    (lambda: W.qwen_u8(6, 2200, seed=105), 4, False),   # 24 u8 rows: the u8 tensor-memory kernel (N = 32)
    (lambda: W.qwen_u8(3, 2200, seed=108), 4, False),   # 12 u8 rows: the same kernel with N = 16
    (lambda: W.make_case("tree_u8_rows64", seed=109, query_lens=[8], past_lens=[1800], num_q_heads=64,
                         num_kv_heads=8, head_dim=128, page_size=16, kv_dtype="u8"), 0, False),  # warp-level u8
    (lambda: W.make_case("tree_d256", seed=106, query_lens=[4, 6], past_lens=[1500, 700], num_q_heads=32,
                         num_kv_heads=16, head_dim=256, page_size=64), 0, False),
    (lambda: W.tiny(seed=107), 1, True),
]


def _gpu_tree(case, mask):
    import torch
    dev = to_device(case)
    d = dims(case, dev)
    kvc = KV_CODE[case.kv_dtype]
    ws = pa.alloc_workspace(d, case.max_context_len, case.sliding_window, kvc)
    tm = torch.from_numpy(mask).cuda()
    pa.forward_tree(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], case.max_context_len, case.scale,
                    case.sliding_window, kvc, dev["out"], d, ws, tm)
    torch.cuda.synchronize()
    bits = pa.device_status(ws)
    plan = pa.plan(d, case.max_context_len, case.sliding_window, kvc,
                   torch.cuda.get_device_properties(0).multi_processor_count)
    return dev["out"].float().cpu().numpy().astype(np.float64), bits, plan.kernel, dev["out"].cpu()


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_tree_verify_matches_the_oracle(idx):
    make, kernel, short = CASES[idx]
    case = make()
    mask = random_tree_masks(case, seed=idx)
    want = oracle.forward(case.q, case.q_dtype, case.k_cache, case.v_cache, case.kv_dtype, case.block_tables,
                          case.past_lens, case.subsequence_begins, num_q_heads=case.num_q_heads,
                          num_kv_heads=case.num_kv_heads, head_dim=case.head_dim, page_size=case.page_size,
                          num_blocks=case.num_blocks, scale=case.scale, sliding_window=case.sliding_window,
                          tree_mask=mask)
    got, bits, k, _ = _gpu_tree(case, mask)
    assert bits == 0
    assert kernel is None or k == kernel, (case.name, k)
    if short:  # O(1) outputs of short contexts: the derived bound (pa_testing.derived_tolerance)
        assert float(np.max(np.abs(got - want) - derived_tolerance(case, want))) <= 0.0
    else:
        assert float(np.max(np.abs(got - want))) <= TOL


@pytest.mark.parametrize("idx", [0, 1, 3])
def test_chain_mask_is_the_plain_verify_bit_for_bit(idx):
    import torch
    case = CASES[idx][0]()
    chain = np.zeros(case.total_tokens, dtype=np.uint8)
    for b in range(case.num_seqs):
        t0 = int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            chain[t0 + i] = (2 << i) - 1
    _, bits, _, raw_tree = _gpu_tree(case, chain)
    assert bits == 0
    dev = to_device(case)
    run_gpu(case, dev=dev)
    assert torch.equal(raw_tree.view(torch.int16), dev["out"].cpu().view(torch.int16))


def test_workspace_size_covers_tree_calls():
    """A tree-mask call with the workspace pa_verify_workspace_size reports
    (which covers the plain and the tree-mask plans), at 32k keys."""
    import torch
    case = W.qwen_u8(6, 32768, seed=106)
    dev = to_device(case)
    d = dims(case, dev)
    kvc = KV_CODE[case.kv_dtype]
    ws = pa.alloc_workspace(d, case.max_context_len, 0, kvc)
    tm = torch.from_numpy(random_tree_masks(case, seed=9)).cuda()
    pa.forward_tree(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], case.max_context_len, case.scale,
                    0, kvc, dev["out"], d, ws, tm)
    torch.cuda.synchronize()
    first = dev["out"].clone()
    big = torch.zeros(ws.numel() * 4, dtype=torch.uint8, device="cuda")
    pa.forward_tree(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], case.max_context_len, case.scale,
                    0, kvc, dev["out"], d, big, tm)
    torch.cuda.synchronize()
    assert pa.device_status(ws) == 0
    assert torch.equal(first.view(torch.int16), dev["out"].view(torch.int16))
