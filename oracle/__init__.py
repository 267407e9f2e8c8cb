"""fp64 CPU oracle for paged verify attention — TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke test and the benchmark's CPU-baseline
leg may import this package.  The product library never imports it, and it
imports nothing from the product: it restates the storage layouts itself.

`pa_oracle.c` holds the definitions: the verify attention (plain C, fp64,
one output row per work item, OpenMP over rows) and the cache update that
precedes it (writing the new tokens' K/V into their pages; u8 caches get a
per-token binary32 min/max quantisation).  This module compiles it with gcc on first use into
``oracle/_build/`` and calls it through ctypes.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, the T-token ≡
T single-token equivalence, a library attention routine, hand-derived golden
values); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "u8": 3}


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (-O2, OpenMP); return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
            ci = ctypes.c_int
            lib.pa_oracle_forward.argtypes = [vp, ci, vp, vp, ci, i32p, i32p, i32p, ci, ci, ci, ci, ci,
                                              ci, ci, ctypes.c_double, ci,
                                              ctypes.POINTER(ctypes.c_double), ci]
            lib.pa_oracle_forward.restype = ci
            lib.pa_oracle_forward_tree.argtypes = [vp, ci, vp, vp, ci, i32p, i32p, i32p, ci, ci, ci, ci, ci,
                                                   ci, ci, ctypes.c_double, ci, vp,
                                                   ctypes.POINTER(ctypes.c_double), ci]
            lib.pa_oracle_forward_tree.restype = ci
            lib.pa_oracle_pages_touched.argtypes = [i32p, i32p, i32p, ci, ci, ci, ci, i32p]
            lib.pa_oracle_pages_touched.restype = ci
            lib.pa_oracle_cache_update.argtypes = [vp, vp, ci, vp, vp, ci, i32p, i32p, i32p, ci, ci, ci, ci, ci, ci]
            lib.pa_oracle_cache_update.restype = ci
            lib.pa_oracle_max_threads.argtypes = []
            lib.pa_oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def max_threads() -> int:
    return int(_load().pa_oracle_max_threads())


def forward(q_raw: np.ndarray, q_dtype: str, k_cache_raw: np.ndarray, v_cache_raw: np.ndarray,
            kv_dtype: str, block_tables, past_lens, subsequence_begins, *, num_q_heads: int,
            num_kv_heads: int, head_dim: int, page_size: int, num_blocks: int, scale: float,
            sliding_window: int = 0, nthreads: int = 0, tree_mask=None) -> np.ndarray:
    """Exact-definition paged verify attention in fp64.  tree_mask (optional,
    uint8 per token, at most 8 new tokens per sequence): bit k set = the token
    sees the sequence's new token k; None = the causal chain.

    Arrays hold the stored bits (f32 values, or uint16 bit patterns for f16 /
    bf16, or the raw bytes of u8 page records).  Returns [total_tokens, Hq, D]
    float64.  Raises ValueError on inconsistent inputs (block id out of range,
    positions beyond the block table).
    """
    lib = _load()
    q_raw = np.ascontiguousarray(q_raw)
    k_cache_raw = np.ascontiguousarray(k_cache_raw)
    v_cache_raw = np.ascontiguousarray(v_cache_raw)
    bt = _i32(block_tables)
    pl = _i32(past_lens)
    sb = _i32(subsequence_begins)
    num_seqs = pl.shape[0]
    assert bt.ndim == 2 and bt.shape[0] == num_seqs and sb.shape[0] == num_seqs + 1
    total_tokens = int(sb[-1])
    out = np.zeros((total_tokens, num_q_heads, head_dim), dtype=np.float64)
    tm = None if tree_mask is None else np.ascontiguousarray(np.asarray(tree_mask, dtype=np.uint8))
    if tm is not None:
        assert tm.shape == (total_tokens,)
    rc = lib.pa_oracle_forward_tree(q_raw.ctypes.data, DTYPE_CODES[q_dtype], k_cache_raw.ctypes.data,
                                    v_cache_raw.ctypes.data, DTYPE_CODES[kv_dtype], _ptr_i32(bt),
                                    _ptr_i32(pl), _ptr_i32(sb), num_seqs, num_q_heads, num_kv_heads,
                                    head_dim, page_size, num_blocks, bt.shape[1], float(scale),
                                    int(sliding_window), None if tm is None else tm.ctypes.data,
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: inconsistent inputs (block id or position out of range)")
    return out


def pages_touched(block_tables, past_lens, subsequence_begins, *, page_size: int,
                  sliding_window: int = 0) -> np.ndarray:
    """[num_seqs, max_blocks_per_seq] int32: physical block id + 1 of every
    logical page the definition reads, 0 for pages it does not read."""
    lib = _load()
    bt = _i32(block_tables)
    pl = _i32(past_lens)
    sb = _i32(subsequence_begins)
    out = np.zeros(bt.shape, dtype=np.int32)
    rc = lib.pa_oracle_pages_touched(_ptr_i32(bt), _ptr_i32(pl), _ptr_i32(sb), pl.shape[0],
                                     page_size, bt.shape[1], int(sliding_window), _ptr_i32(out))
    if rc != 0:
        raise ValueError("oracle: key range runs past the block table")
    return out


def cache_update(k_new_raw: np.ndarray, v_new_raw: np.ndarray, src_dtype: str, k_cache_raw: np.ndarray,
                 v_cache_raw: np.ndarray, kv_dtype: str, block_tables, past_lens, subsequence_begins, *,
                 num_kv_heads: int, head_dim: int, page_size: int, num_blocks: int):
    """The cache-update definition (pa_oracle.c): returns new copies of the two
    caches with the new tokens written.  Arrays hold stored bits, as in
    forward(); k_new / v_new are [total_tokens, Hkv, D].  Raises ValueError on
    inconsistent inputs."""
    lib = _load()
    k_new_raw = np.ascontiguousarray(k_new_raw)
    v_new_raw = np.ascontiguousarray(v_new_raw)
    kc = np.array(k_cache_raw, copy=True, order="C")
    vc = np.array(v_cache_raw, copy=True, order="C")
    bt = _i32(block_tables)
    pl = _i32(past_lens)
    sb = _i32(subsequence_begins)
    rc = lib.pa_oracle_cache_update(k_new_raw.ctypes.data, v_new_raw.ctypes.data, DTYPE_CODES[src_dtype],
                                    kc.ctypes.data, vc.ctypes.data, DTYPE_CODES[kv_dtype], _ptr_i32(bt),
                                    _ptr_i32(pl), _ptr_i32(sb), pl.shape[0], num_kv_heads, head_dim, page_size,
                                    num_blocks, bt.shape[1])
    if rc != 0:
        raise ValueError("oracle: inconsistent cache-update inputs")
    return kc, vc
