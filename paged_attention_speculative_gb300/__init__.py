"""paged_attention_speculative_gb300 — paged attention for speculative-decoding
verification on GB300 (sm_103a).

A thin ctypes binding over ``libpa_verify.so`` (C ABI in
``include/pa_verify.h``).  The binding only marshals arguments: every step of
the verify path runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing, loading raises.

Entry points mirror the C ABI:
  forward / forward_traced / forward_tree / partition / combine / workspace_size / plan /
  device_status / status_string, forward_mixed / forward_mixed_tree (verify
  steps and prefill chunks in one call), and cache_update (the step before
  the verify: the new tokens' K/V written into their pages)
Tensors are torch CUDA tensors (torch supplies device memory and streams).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["PA_F32", "PA_F16", "PA_BF16", "PA_U8", "PaDims", "PaPlan", "load_library", "library_path",
           "forward", "forward_traced", "partition", "combine", "workspace_size", "plan", "device_status",
           "status_string", "dims_for", "cache_update", "forward_tree", "forward_mixed", "forward_mixed_tree",
           "PaVerifyError"]

PA_F32, PA_F16, PA_BF16, PA_U8 = 0, 1, 2, 3
PA_MAX_QUERY_LEN = 8
STATUS_BITS = {0x1: "QUERY_LEN", 0x2: "CONTEXT", 0x4: "BLOCK_ID", 0x8: "BEGINS", 0x10: "PAST_LEN",
               0x20: "ROWS", 0x40: "TIMEOUT"}
EXPORTED = ["pa_verify_workspace_size", "pa_verify_plan", "pa_verify_forward", "pa_verify_forward_traced",
            "pa_verify_partition", "pa_verify_combine", "pa_verify_get_device_status", "pa_verify_status_string",
            "pa_verify_forward_no_alloc", "pa_cache_update", "pa_verify_forward_tree", "pa_mixed_workspace_size",
            "pa_forward_mixed", "pa_forward_mixed_tree"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class PaVerifyError(RuntimeError):
    pass


class PaDims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32), ("q_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int)]


class PaPlan(ctypes.Structure):
    _fields_ = [("num_partitions", ctypes.c_int32), ("part_tokens", ctypes.c_int32),
                ("stage_keys", ctypes.c_int32), ("row_tiles", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("ctas", ctypes.c_int32), ("smem_bytes", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libpa_verify.so")


def load_library():
    """Load libpa_verify.so (built by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise PaVerifyError(f"libpa_verify.so not built ({path}); run paged_attention_speculative_gb300.build")
        try:
            import torch  # noqa: F401  (load torch's libcudart.so.13 first so both share it)
        except ImportError:
            pass
        lib = ctypes.CDLL(path)
        vp, i32, i32p, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t
        dp = ctypes.POINTER(PaDims)
        fwd = [vp, vp, vp, vp, vp, vp, i32, ctypes.c_float, i32, ctypes.c_int, vp, dp, vp, sz, vp]
        lib.pa_verify_workspace_size.argtypes = [dp, i32, i32, ctypes.c_int]
        lib.pa_verify_workspace_size.restype = sz
        lib.pa_verify_plan.argtypes = [dp, i32, i32, ctypes.c_int, i32, ctypes.POINTER(PaPlan)]
        lib.pa_verify_plan.restype = ctypes.c_int
        lib.pa_verify_forward.argtypes = fwd
        lib.pa_verify_forward.restype = ctypes.c_int
        lib.pa_verify_forward_traced.argtypes = fwd + [vp]
        lib.pa_verify_forward_traced.restype = ctypes.c_int
        lib.pa_verify_partition.argtypes = fwd
        lib.pa_verify_partition.restype = ctypes.c_int
        lib.pa_verify_combine.argtypes = [vp, vp, i32, i32, ctypes.c_int, vp, dp, vp, sz, vp]
        lib.pa_verify_combine.restype = ctypes.c_int
        lib.pa_verify_get_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.pa_verify_get_device_status.restype = ctypes.c_int
        lib.pa_verify_forward_no_alloc.argtypes = fwd[:12] + [vp]
        lib.pa_verify_forward_no_alloc.restype = ctypes.c_int
        lib.pa_verify_forward_tree.argtypes = fwd[:14] + [vp, vp]
        lib.pa_verify_forward_tree.restype = ctypes.c_int
        lib.pa_mixed_workspace_size.argtypes = [dp, i32, i32, ctypes.c_int]
        lib.pa_mixed_workspace_size.restype = sz
        lib.pa_forward_mixed.argtypes = fwd
        lib.pa_forward_mixed.restype = ctypes.c_int
        lib.pa_forward_mixed_tree.argtypes = fwd[:14] + [vp, vp]
        lib.pa_forward_mixed_tree.restype = ctypes.c_int
        lib.pa_cache_update.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, vp, dp,
                                        vp, vp]
        lib.pa_cache_update.restype = ctypes.c_int
        lib.pa_verify_status_string.argtypes = [ctypes.c_int]
        lib.pa_verify_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().pa_verify_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise PaVerifyError(f"{what} failed: {rc} ({status_string(rc)})")


def _torch_dtype_code(dt) -> int:
    import torch
    table = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_U8}
    if dt not in table:
        raise PaVerifyError(f"unsupported dtype {dt}")
    return table[dt]


def dims_for(q, k_cache, block_tables, past_lens, out, *, num_kv_heads: int | None = None,
             page_size: int | None = None, head_dim: int | None = None) -> PaDims:
    """pa_dims from the tensors: q [T, Hq, D], block_tables [B, W], out [T, Hq, D];
    k_cache [nb, Hkv, ps, D] (16-bit / f32) or u8 records [nb, Hkv, ps*(D+4)]
    (then page_size is required)."""
    tt, hq, d = q.shape
    if head_dim is not None:
        d = head_dim
    if k_cache.dim() == 4:
        nb, hkv, ps, _ = k_cache.shape
    else:
        nb, hkv, _ = k_cache.shape
        if page_size is None:
            raise PaVerifyError("page_size is required for u8 page records")
        ps = page_size
    if num_kv_heads is not None:
        hkv = num_kv_heads
    if page_size is not None:
        ps = page_size
    return PaDims(num_seqs=past_lens.shape[0], total_tokens=tt, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                  page_size=ps, num_blocks=nb, max_blocks_per_seq=block_tables.shape[1],
                  q_dtype=_torch_dtype_code(q.dtype), out_dtype=_torch_dtype_code(out.dtype))


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def workspace_size(dims: PaDims, max_context_len: int, sliding_window: int, kv_dtype: int) -> int:
    return int(load_library().pa_verify_workspace_size(ctypes.byref(dims), int(max_context_len),
                                                       int(sliding_window), int(kv_dtype)))


def plan(dims: PaDims, max_context_len: int, sliding_window: int, kv_dtype: int, num_sms: int) -> PaPlan:
    p = PaPlan()
    _check(load_library().pa_verify_plan(ctypes.byref(dims), int(max_context_len), int(sliding_window),
                                         int(kv_dtype), int(num_sms), ctypes.byref(p)), "pa_verify_plan")
    return p


def alloc_workspace(dims: PaDims, max_context_len: int, sliding_window: int, kv_dtype: int, device=None):
    """A zeroed workspace tensor of the size pa_verify_workspace_size asks for."""
    import torch
    n = workspace_size(dims, max_context_len, sliding_window, kv_dtype)
    if n == 0:
        raise PaVerifyError("pa_verify_workspace_size rejected the arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _fwd_args(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
              sliding_window, kv_dtype, out, dims, workspace, stream):
    return (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(past_lens), _ptr(subsequence_begins),
            int(max_context_len), float(scale), int(sliding_window), int(kv_dtype), _ptr(out), ctypes.byref(dims),
            _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream_ptr(stream))


def forward(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
            sliding_window, kv_dtype, out, dims: PaDims, workspace, stream=None):
    """pa_verify_forward: writes out [T, Hq, D]; asynchronous on `stream`."""
    _check(load_library().pa_verify_forward(*_fwd_args(q, k_cache, v_cache, block_tables, past_lens,
                                                       subsequence_begins, max_context_len, scale, sliding_window,
                                                       kv_dtype, out, dims, workspace, stream)), "pa_verify_forward")
    return out


def forward_traced(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                   sliding_window, kv_dtype, out, dims: PaDims, workspace, trace, stream=None):
    """pa_verify_forward_traced: also adds (block id + 1) per fetched page into trace."""
    _check(load_library().pa_verify_forward_traced(*_fwd_args(q, k_cache, v_cache, block_tables, past_lens,
                                                              subsequence_begins, max_context_len, scale,
                                                              sliding_window, kv_dtype, out, dims, workspace,
                                                              stream), _ptr(trace)), "pa_verify_forward_traced")
    return out


def forward_tree(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                 sliding_window, kv_dtype, out, dims: PaDims, workspace, tree_mask, stream=None):
    """pa_verify_forward_tree: like forward, with the new tokens seeing each
    other through tree_mask (uint8 device tensor [total_tokens], bit k = sees
    its sequence's new token k)."""
    args = _fwd_args(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                     sliding_window, kv_dtype, out, dims, workspace, stream)
    _check(load_library().pa_verify_forward_tree(*args[:14], _ptr(tree_mask), args[14]), "pa_verify_forward_tree")
    return out


def mixed_workspace_size(dims: PaDims, max_context_len: int, sliding_window: int, kv_dtype: int) -> int:
    return int(load_library().pa_mixed_workspace_size(ctypes.byref(dims), int(max_context_len),
                                                      int(sliding_window), int(kv_dtype)))


def alloc_mixed_workspace(dims: PaDims, max_context_len: int, sliding_window: int, kv_dtype: int, device=None):
    """A zeroed workspace tensor of the size pa_mixed_workspace_size asks for."""
    import torch
    n = mixed_workspace_size(dims, max_context_len, sliding_window, kv_dtype)
    if n == 0:
        raise PaVerifyError("pa_mixed_workspace_size rejected the arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def forward_mixed(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                  sliding_window, kv_dtype, out, dims: PaDims, workspace, stream=None):
    """pa_forward_mixed: verify steps (T_b <= 8) and prefill chunks (T_b > 8)
    in one call; the workspace from alloc_mixed_workspace."""
    _check(load_library().pa_forward_mixed(*_fwd_args(q, k_cache, v_cache, block_tables, past_lens,
                                                      subsequence_begins, max_context_len, scale, sliding_window,
                                                      kv_dtype, out, dims, workspace, stream)), "pa_forward_mixed")
    return out


def forward_mixed_tree(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                       sliding_window, kv_dtype, out, dims: PaDims, workspace, tree_mask, stream=None):
    """pa_forward_mixed_tree: forward_mixed with the verify steps' new tokens
    seeing each other through tree_mask (prefill chunks stay causal)."""
    args = _fwd_args(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
                     sliding_window, kv_dtype, out, dims, workspace, stream)
    _check(load_library().pa_forward_mixed_tree(*args[:14], _ptr(tree_mask), args[14]), "pa_forward_mixed_tree")
    return out


def partition(q, k_cache, v_cache, block_tables, past_lens, subsequence_begins, max_context_len, scale,
              sliding_window, kv_dtype, out, dims: PaDims, workspace, stream=None):
    _check(load_library().pa_verify_partition(*_fwd_args(q, k_cache, v_cache, block_tables, past_lens,
                                                         subsequence_begins, max_context_len, scale, sliding_window,
                                                         kv_dtype, out, dims, workspace, stream)),
           "pa_verify_partition")


def combine(past_lens, subsequence_begins, max_context_len, sliding_window, kv_dtype, out, dims: PaDims, workspace,
            stream=None):
    _check(load_library().pa_verify_combine(_ptr(past_lens), _ptr(subsequence_begins), int(max_context_len),
                                            int(sliding_window), int(kv_dtype), _ptr(out), ctypes.byref(dims),
                                            _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                            _stream_ptr(stream)), "pa_verify_combine")


def device_status(workspace, stream=None) -> int:
    """Synchronise the stream, read and clear the sticky device status bits."""
    bits = ctypes.c_uint32(0)
    _check(load_library().pa_verify_get_device_status(_ptr(workspace), _stream_ptr(stream), ctypes.byref(bits)),
           "pa_verify_get_device_status")
    return int(bits.value)


def cache_update(k_new, v_new, k_cache, v_cache, block_tables, past_lens, subsequence_begins, dims: PaDims,
                 status=None, stream=None):
    """pa_cache_update: write the new tokens' K / V ([total_tokens, Hkv, D],
    f32 / f16 / bf16) into their pages of k_cache / v_cache (float caches, or
    uint8 page records); asynchronous on `stream`.  `status` is an optional
    int32 / uint32 device tensor of one element that collects PA_STATUS_* bits."""
    kv = _torch_dtype_code(k_cache.dtype)
    _check(load_library().pa_cache_update(_ptr(k_new), _ptr(v_new), _torch_dtype_code(k_new.dtype), _ptr(k_cache),
                                          _ptr(v_cache), int(kv), _ptr(block_tables), _ptr(past_lens),
                                          _ptr(subsequence_begins), ctypes.byref(dims), _ptr(status),
                                          _stream_ptr(stream)), "pa_cache_update")
