"""Mixed batches on the GPU (pa_forward_mixed, through the C ABI): verify
steps (T_b <= 8) on the split-KV kernels and prefill chunks (T_b > 8) on the
prefill tile kernel, in one call, against the oracle (whose causal rule holds
for any number of new tokens).  Cases cover the query-head group sizes the
tiles handle (G = 1, 2, 4, 6, 8: blocks of 128 / G tokens, or 256 / G in the
two-tile blocks a tuning override selects, ragged last blocks), windows,
f16 / bf16 / fp32
caches, large pages, keys split into pieces (few blocks at long context),
and device errors in a prefill chunk; a mixed call with no prefill chunk is
pa_verify_forward bit for bit."""
import numpy as np
import pytest

import oracle
import paged_attention_speculative_gb300 as pa
from paged_attention_speculative_gb300 import workloads as W

from pa_testing import KV_CODE, TOL, derived_tolerance, dims, max_abs_err, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


def run_mixed(case, dev=None, max_context_len=None):
    import torch
    dev = dev or to_device(case)
    d = dims(case, dev)
    kvc = KV_CODE[case.kv_dtype]
    mcl = max_context_len or case.max_context_len
    ws = pa.alloc_mixed_workspace(d, mcl, case.sliding_window, kvc)
    pa.forward_mixed(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], mcl, case.scale,
                     case.sliding_window, kvc, dev["out"], d, ws)
    torch.cuda.synchronize()
    return dev["out"].float().cpu().numpy().astype(np.float64), pa.device_status(ws), dev["out"].cpu()


def mk(name, seed, ql, pl, hq, hkv, d=128, ps=16, **kw):
    return lambda: W.make_case(name, seed=seed, query_lens=ql, past_lens=pl, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=d, page_size=ps, **kw)


CASES = [
    # (factory, derived bound: short contexts with O(1) outputs)
    (mk("prefill_g4", 70, [100], [1000], 32, 8), False),
    (mk("mixed_g4", 71, [4, 200, 1, 0, 37, 8, 9], [3000, 500, 1500, 10, 0, 700, 2000], 32, 8), True),
    (mk("mixed_g8", 72, [8, 300], [20000, 20000], 64, 8), False),
    (mk("mixed_win", 73, [50, 3, 130], [2000, 900, 64], 32, 8, sliding_window=300), True),
    (mk("mixed_f16_d64_g2", 74, [150, 2], [400, 800], 8, 4, d=64, q_dtype="f16", kv_dtype="f16"), True),
    (mk("prefill_g1", 75, [260], [700], 8, 8), False),
    (mk("prefill_g6", 76, [50, 5], [300, 90], 24, 4), True),
    (mk("mixed_f32", 77, [3, 20], [40, 10], 4, 2, d=64, q_dtype="f32", kv_dtype="f32"), True),
    (mk("prefill_ps128", 78, [70, 2], [1000, 130], 32, 8, ps=128), False),
    (mk("prefill_ps8_win1", 79, [40], [100], 8, 2, ps=8, sliding_window=1), True),
    # many blocks (several waves of 128-row blocks), head_dim 64
    (mk("prefill_many_blocks", 85, [1200, 2], [100, 300], 64, 32, d=64), True),
    # few blocks at long context: the blocks' keys split into pieces merged by
    # the prefill combine (2 pieces; 2 inside a window; 6 for the long
    # chunk beside a short one at past 0, which stays whole; 4 at head_dim 64)
    (mk("split_small_chunk", 90, [24, 4, 1], [12000, 9000, 500], 32, 8), False),
    (mk("split_window", 91, [40, 2], [30000, 100], 32, 8, sliding_window=9000), False),
    (mk("split_short_and_long", 92, [20, 60, 3], [0, 40000, 800], 32, 8), True),
    (mk("split_f16_d64", 93, [30], [16384], 8, 4, d=64, q_dtype="f16", kv_dtype="f16"), False),
    # six real blocks: 3 of the 4 pieces the host provides for
    (mk("split_fewer_than_launched", 94, [40, 40, 40], [20000, 20000, 20000], 32, 8), False),
]
# pieces the host provides for (the grid's z extent); the kernels use as many
# as fit in one wave for the blocks the batch really has
SPLIT = {"split_small_chunk": 2, "split_window": 2, "split_short_and_long": 9, "split_f16_d64": 4,
         "split_fewer_than_launched": 4}


def prefill_pieces(case):
    """Key pieces of the case's prefill blocks, read back from the size of
    the mixed workspace: the verify part's bytes plus total_tokens x Hq x
    pieces partial rows when the keys are split."""
    import torch
    a256 = lambda x: (x + 255) // 256 * 256
    d = dims(case, to_device(case))
    kvc = KV_CODE[case.kv_dtype]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = pa.plan(d, case.max_context_len, case.sliding_window, kvc, sms)
    rows = case.num_seqs * 8 * case.num_q_heads * p.num_partitions
    extra = pa.mixed_workspace_size(d, case.max_context_len, case.sliding_window, kvc) - (
        256 + a256(rows * case.head_dim * 4) + 2 * a256(rows * 4))
    if extra == 0:
        return 1
    prow = case.total_tokens * case.num_q_heads
    for S in range(2, 33):
        if a256(prow * S * case.head_dim * 4) + 2 * a256(prow * S * 4) == extra:
            return S
    raise AssertionError(f"workspace tail of {extra} bytes matches no piece count")


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_mixed_matches_the_oracle(idx):
    make, derived = CASES[idx]
    case = make()
    assert prefill_pieces(case) == SPLIT.get(case.name, 1)
    got, bits, _ = run_mixed(case)
    assert bits == 0, f"device status {bits:#x}"
    want = run_oracle(case)
    err = max_abs_err(got, want)
    if derived:
        worst = float(np.max(np.abs(got - want) - derived_tolerance(case, want)))
        assert worst <= 0.0, f"{case.name}: exceeds the derived bound by {worst:.3e} (max abs {err:.3e})"
    else:
        assert err <= TOL, f"{case.name}: max abs err {err:.3e}"


_TWO_TILE_CHILD = r"""
import sys, numpy as np
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from paged_attention_speculative_gb300 import workloads as W
import test_gpu_mixed as M
from pa_testing import derived_tolerance, run_oracle
for name, seed, ql, pl, hq, hkv, d in (("two_tile_g4", 87, [300, 3], [2000, 700], 32, 8, 128),
                                        ("two_tile_g2_d64", 88, [260], [5000], 16, 8, 64)):
    case = W.make_case(name, seed=seed, query_lens=ql, past_lens=pl, num_q_heads=hq, num_kv_heads=hkv,
                       head_dim=d, page_size=16)
    got, bits, _ = M.run_mixed(case)
    assert bits == 0, bits
    want = run_oracle(case)
    assert float(np.max(np.abs(got - want) - derived_tolerance(case, want))) <= 0.0, name
print("two-tile ok")
"""


def test_two_tile_blocks_by_override():
    """Blocks of 256 rows (two tiles ping-ponging on shared K/V stages) are
    not the default (128-row blocks measured faster); PA_PREFILL_ROWS=256
    selects them, read once per process, so a child process checks them
    against the oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PA_PREFILL_ROWS="256")
    r = subprocess.run([sys.executable, "-c", _TWO_TILE_CHILD, root], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "two-tile ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.slow
def test_mixed_full_size():
    """A prefill chunk of 130 tokens and three T=4 verify steps at 32k keys
    (Qwen-like heads)."""
    case = W.make_case("mixed_32k", seed=80, query_lens=[4, 130, 4, 4], past_lens=[32768, 32768, 30000, 32000],
                       num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    assert prefill_pieces(case) == 4
    got, bits, _ = run_mixed(case)
    assert bits == 0
    assert max_abs_err(got, run_oracle(case)) <= TOL


def test_mixed_without_prefill_is_the_verify_call_bit_for_bit():
    import torch
    case = W.make_case("no_prefill", seed=81, query_lens=[4, 1, 8, 3], past_lens=[5000, 3000, 4500, 100],
                       num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _, bits, raw = run_mixed(case)
    assert bits == 0
    dev = to_device(case)
    run_gpu(case, dev=dev)
    assert torch.equal(raw.view(torch.int16), dev["out"].cpu().view(torch.int16))


def test_prefill_chunk_equals_its_tokens_as_decodes():
    """The pages' equivalence at prefill length: token i of a 40-token chunk
    equals a single-token decode at past_len L + i (within the tolerance)."""
    case = W.make_case("eq", seed=82, query_lens=[40], past_lens=[3000], num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=16)
    multi, bits, _ = run_mixed(case)
    assert bits == 0
    for i in (0, 17, 39):
        single = W.Case(**{**case.__dict__, "q": case.q[i:i + 1].copy(), "past_lens": np.array([3000 + i], np.int32),
                           "subsequence_begins": np.array([0, 1], np.int32), "name": f"single{i}"})
        got, bits, _ = run_gpu(single)
        assert bits == 0
        assert np.max(np.abs(got[0] - multi[i])) <= TOL


def test_bad_block_id_in_a_prefill_chunk_sets_the_status():
    case = W.make_case("bad", seed=83, query_lens=[3, 60], past_lens=[500, 700], num_q_heads=32, num_kv_heads=8,
                       head_dim=128, page_size=16)
    bt = case.block_tables.copy()
    bt[1, 10] = case.num_blocks + 3
    bad = W.Case(**{**case.__dict__, "block_tables": bt})
    got, bits, _ = run_mixed(bad)
    assert bits & 0x4  # PA_STATUS_BLOCK_ID
    good = run_oracle(case)
    # the verify step is untouched; the chunk's tiles that read the bad page are zero
    assert max_abs_err(got[:3], good[:3]) <= TOL


def test_bad_block_id_in_a_split_prefill_chunk_zeroes_its_rows():
    """A bad id read by one key piece poisons that piece's partial rows; the
    prefill combine zeroes the rows, the verify step is untouched."""
    case = W.make_case("bad_split", seed=86, query_lens=[3, 40], past_lens=[500, 12000], num_q_heads=32,
                       num_kv_heads=8, head_dim=128, page_size=16)
    assert prefill_pieces(case) == 2
    bt = case.block_tables.copy()
    bt[1, 600] = case.num_blocks + 3  # keys 9600..9615: the second piece of every block
    bad = W.Case(**{**case.__dict__, "block_tables": bt})
    got, bits, _ = run_mixed(bad)
    assert bits & 0x4  # PA_STATUS_BLOCK_ID
    assert max_abs_err(got[:3], run_oracle(case)[:3]) <= TOL
    assert np.all(got[3:] == 0.0)


def test_context_overflow_in_a_prefill_chunk_sets_the_status():
    case = W.make_case("ctx", seed=84, query_lens=[2, 40], past_lens=[100, 200], num_q_heads=8, num_kv_heads=2,
                       head_dim=128, page_size=16)
    got, bits, _ = run_mixed(case, max_context_len=220)
    assert bits & 0x2  # PA_STATUS_CONTEXT
    assert np.all(got[2:] == 0.0)


def _sub_case(case, seqs):
    """The sub-batch of `case` holding sequences `seqs` (same caches and block
    tables), with the token map back into the full batch."""
    import dataclasses
    sb = case.subsequence_begins
    rows, begins = [], [0]
    for b in seqs:
        rows.extend(range(int(sb[b]), int(sb[b + 1])))
        begins.append(begins[-1] + int(sb[b + 1] - sb[b]))
    sub = dataclasses.replace(case, q=case.q[rows], block_tables=case.block_tables[list(seqs)],
                              past_lens=case.past_lens[list(seqs)],
                              subsequence_begins=np.asarray(begins, dtype=np.int32))
    return sub, rows


@pytest.mark.parametrize("idx", [1, 3, 7])
def test_mixed_tree_masks(idx):
    """pa_forward_mixed_tree: the verify steps' draft tokens see each other
    through random tree masks, the prefill chunks stay causal (their mask
    entries are set to all ones and must not be read).  Expected: the
    oracle's tree definition on the verify sequences, its causal definition
    on the prefill ones."""
    import torch
    make, derived = CASES[idx]
    case = make()
    # masks for the verify sequences only; prefill tokens get 0xff (ignored)
    rng = np.random.default_rng(400 + idx)
    mask = np.full(case.total_tokens, 0xFF, dtype=np.uint8)
    verify = [b for b in range(case.num_seqs) if 0 < int(case.query_lens[b]) <= 8]
    prefill = [b for b in range(case.num_seqs) if int(case.query_lens[b]) > 8]
    for b in verify:
        t0 = int(case.subsequence_begins[b])
        for i in range(int(case.query_lens[b])):
            parent = -1 if i == 0 else int(rng.integers(-1, i))
            mask[t0 + i] = (1 << i) | (mask[t0 + parent] if parent >= 0 else 0)
    dev = to_device(case)
    d = dims(case, dev)
    kvc = KV_CODE[case.kv_dtype]
    ws = pa.alloc_mixed_workspace(d, case.max_context_len, case.sliding_window, kvc)
    pa.forward_mixed_tree(dev["q"], dev["k"], dev["v"], dev["bt"], dev["pl"], dev["sb"], case.max_context_len,
                          case.scale, case.sliding_window, kvc, dev["out"], d, ws, torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    assert pa.device_status(ws) == 0
    got = dev["out"].float().cpu().numpy().astype(np.float64)
    want = np.zeros_like(got)
    for seqs, tree in ((verify, True), (prefill, False)):
        if not seqs:
            continue
        sub, rows = _sub_case(case, seqs)
        kw = dict(num_q_heads=sub.num_q_heads, num_kv_heads=sub.num_kv_heads, head_dim=sub.head_dim,
                  page_size=sub.page_size, num_blocks=sub.num_blocks, scale=sub.scale,
                  sliding_window=sub.sliding_window)
        want[rows] = oracle.forward(sub.q, sub.q_dtype, sub.k_cache, sub.v_cache, sub.kv_dtype, sub.block_tables,
                                    sub.past_lens, sub.subsequence_begins, tree_mask=mask[rows] if tree else None,
                                    **kw)
    err = max_abs_err(got, want)
    if derived:
        worst = float(np.max(np.abs(got - want) - derived_tolerance(case, want)))
        assert worst <= 0.0, f"{case.name}: exceeds the derived bound by {worst:.3e} (max abs {err:.3e})"
    else:
        assert err <= TOL, f"{case.name}: max abs err {err:.3e}"
