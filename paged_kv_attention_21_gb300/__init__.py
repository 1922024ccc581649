"""Attention over a paged KV cache, hand-written CUDA for GB300 (sm_103a).

A thin ctypes binding over ``libpkv.so`` (C ABI in ``include/pkv.h``).  Each
function carries the C entry point's name and only marshals arguments: torch
tensors become pointers (device memory, or pinned host memory where the C
declaration allows it), the current torch stream becomes the launch stream,
and a non-OK status raises :class:`PkvError` with the library's message.  Every step of the computation runs in the library's kernels; if the
library is missing the call fails loudly -- there is no fallback.

PyTorch is used here for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np

from . import build as _build

KV_BF16 = 0
KV_FP8_E4M3 = 1
DESC_PREFETCH_KV = 0x1  # pkv_cache_desc.flags: see PKV_DESC_PREFETCH_KV in pkv.h
DESC_INDEPENDENT = 0x2  # pkv_cache_desc.flags: see PKV_DESC_INDEPENDENT in pkv.h
DEVERR_BLOCK_ID = 0x1
DEVERR_POSITION = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_LENGTH = 0x8

_STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
           3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA"}


class PkvError(RuntimeError):
    """A libpkv call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS.get(status, str(status)), message))
        self.status = status


class CacheDesc(ctypes.Structure):
    """pkv_cache_desc."""

    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("ring_blocks", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


def make_desc(*, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
              kv_dtype=KV_BF16, block_size=16, ring_blocks=0, flags=0) -> CacheDesc:
    """flags: DESC_PREFETCH_KV (see pkv.h) or 0."""
    if isinstance(kv_dtype, str):
        kv_dtype = KV_FP8_E4M3 if kv_dtype.startswith("fp8") else KV_BF16
    return CacheDesc(int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                     int(kv_dtype), int(max_blocks_per_seq), int(num_blocks), int(ring_blocks),
                     int(flags))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libpkv.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError("libpkv.so is not built (%s); run __graft_entry__.build()" % path)
        lib = ctypes.CDLL(path)
        P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        D = ctypes.POINTER(CacheDesc)
        sig = {
            "pkv_cache_bytes": (ctypes.c_uint64, [D]),
            "pkv_append_rope": (ctypes.c_int, [D, P, P, P, P, P, i32, P, P, i32, P, P, P, P, i32, P]),
            "pkv_rope_cos_sin_table": (ctypes.c_int, [f32, i32, i32, P]),
            "pkv_gather_kv": (ctypes.c_int, [D, P, P, P, P, i32, i64, P, P]),
            "pkv_decode_attention": (ctypes.c_int, [D, P, P, P, P, P, P, P, i32, i32, f32, i32, P,
                                                    i32, P, P, P, ctypes.c_size_t, P]),
            "pkv_decode_step": (ctypes.c_int, [D, P, P, P, P, i32, P, P, P, P, P, P, i32, i32, f32,
                                               i32, P, i32, P, P, P, ctypes.c_size_t, P]),
            "pkv_decode_workspace_size": (ctypes.c_size_t, [D, i32, i32, i32, i32]),
            "pkv_decode_plan": (ctypes.c_int, [D, i32, i32, i32, i32, P, P]),
            "pkv_prefill_attention_ragged": (ctypes.c_int, [D, P, P, P, P, P, P, P, P, i32, i32,
                                                            P, P, f32, i32, i32, P, P, P,
                                                            ctypes.c_size_t, P]),
            "pkv_prefill_workspace_size": (ctypes.c_size_t, [D, i32, i32]),
            "pkv_decode_attention_static": (ctypes.c_int, [D, P, P, P, P, P, P, P, i32, i32, f32,
                                                           i32, P, i32, P, P, P]),
            "pkv_merge_states": (ctypes.c_int, [P, P, i32, i32, i32, i32, P, P, P]),
            "pkv_cascade_workspace_size": (ctypes.c_size_t, [D, i32, i32, i32, i32, i32]),
            "pkv_cascade_decode": (ctypes.c_int, [D, P, P, P, P, P, i32, P, P, P, P, P, i32, P, P, i32,
                                                  f32, i32, P, P, P, ctypes.c_size_t, P]),
            "pkv_copy_blocks": (ctypes.c_int, [D, P, P, P, P, i32, P]),
            "pkv_last_error": (ctypes.c_char_p, []),
            "pkv_device_errors": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), i32]),
            "pkv_test_inject_wait_timeout": (ctypes.c_int, [i32, ctypes.c_uint32]),
            "pkv_prefill_ring_commit": (ctypes.c_int, [D, P, P, P, P, P, P, P, P, P, P, i32, i32, P, P,
                                                       f32, i32, P, P, P, ctypes.c_size_t, P]),
            "pkv_prefill_ring_workspace_size": (ctypes.c_size_t, [D, i32, i32, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        raise PkvError(status, load_library().pkv_last_error().decode(errors="replace"))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------ entry points --

def pkv_cache_bytes(desc: CacheDesc) -> int:
    return int(load_library().pkv_cache_bytes(ctypes.byref(desc)))


def pkv_rope_cos_sin_table(theta: float, rotary_dim: int, max_pos: int) -> np.ndarray:
    """Host fp32 [max_pos][rotary_dim/2][2] (cos, sin) table."""
    out = np.empty((max_pos, rotary_dim // 2, 2), dtype=np.float32)
    _check(load_library().pkv_rope_cos_sin_table(float(theta), int(rotary_dim), int(max_pos),
                                                 _ptr(out)))
    return out


def pkv_append_rope(desc, k_cache, v_cache, block_tables, token_to_seq, positions, k_new, v_new,
                    q=None, cos_sin=None, k_scale=None, v_scale=None, num_seqs=None, stream=None):
    num_seqs = block_tables.shape[0] if num_seqs is None else num_seqs
    max_pos = 0 if cos_sin is None else cos_sin.shape[0]
    _check(load_library().pkv_append_rope(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), int(num_seqs), _ptr(token_to_seq), _ptr(positions),
        int(positions.shape[0]), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(cos_sin), int(max_pos),
        _stream(stream)))


def pkv_gather_kv(desc, cache, block_tables, context_lens, cu_context_lens, total_tokens, out,
                  stream=None):
    _check(load_library().pkv_gather_kv(
        ctypes.byref(desc), _ptr(cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(cu_context_lens), int(context_lens.shape[0]), int(total_tokens), _ptr(out),
        _stream(stream)))


def pkv_copy_blocks(desc, k_cache, v_cache, src_blocks, dst_blocks, stream=None):
    """Copy-on-write: block dst_blocks[i] of both pools receives block src_blocks[i]."""
    _check(load_library().pkv_copy_blocks(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(src_blocks), _ptr(dst_blocks),
                                          int(src_blocks.shape[0]), _stream(stream)))


def pkv_decode_workspace_size(desc, num_seqs, max_context_len, window=-1, chunk_blocks=0) -> int:
    return int(load_library().pkv_decode_workspace_size(ctypes.byref(desc), int(num_seqs),
                                                        int(max_context_len), int(window),
                                                        int(chunk_blocks)))


def pkv_decode_plan(desc, num_seqs, max_context_len, window=-1, num_sms=0):
    """Host planner: returns (chunk_blocks, max_splits)."""
    c, s = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().pkv_decode_plan(ctypes.byref(desc), int(num_seqs), int(max_context_len),
                                          int(window), int(num_sms), ctypes.byref(c),
                                          ctypes.byref(s)))
    return c.value, s.value


def pkv_decode_attention(desc, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                         sm_scale, out, lse=None, workspace=None, window=-1, chunk_blocks=0,
                         k_scale=None, v_scale=None, sinks=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().pkv_decode_attention(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(context_lens), int(context_lens.shape[0]), int(max_context_len),
        float(sm_scale), int(window), _ptr(sinks), int(chunk_blocks), _ptr(out), _ptr(lse),
        _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_decode_step(desc, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                    max_context_len, sm_scale, out, lse=None, workspace=None, cos_sin=None,
                    window=-1, chunk_blocks=0, k_scale=None, v_scale=None, sinks=None, stream=None):
    """One decode step of one layer in one launch: append each sequence's new
    token (k_new, v_new; RoPE'd with cos_sin) at context_lens - 1, rotate q
    (read only), and attend -- as pkv_append_rope then pkv_decode_attention.

    q, k_new, v_new, block_tables, context_lens, the scales, sinks, out and
    lse may also be pinned CPU tensors (``tensor.pin_memory()``): the kernel
    reads and writes them over the host link itself.  The caches, workspace
    and cos_sin stay on the GPU."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    max_pos = 0 if cos_sin is None else int(cos_sin.shape[0])
    _check(load_library().pkv_decode_step(
        ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cos_sin), max_pos,
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
        _ptr(context_lens), int(context_lens.shape[0]), int(max_context_len), float(sm_scale),
        int(window), _ptr(sinks), int(chunk_blocks), _ptr(out), _ptr(lse), _ptr(workspace),
        ws_bytes, _stream(stream)))


class BoundCall:
    """A C-ABI call with its arguments marshalled once.  The tensors are bound
    by address and kept alive here: write new contents into the same tensors
    and call again (the persistent-buffer pattern of a serving loop).  Each
    call returns after the launch, like the unbound function."""

    __slots__ = ("_fn", "_args", "_keep")

    def __init__(self, fn, args, keep):
        self._fn = fn
        self._args = args
        self._keep = keep

    def __call__(self):
        st = self._fn(*self._args)
        if st != 0:
            _check(st)


def bind_decode_step(desc, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                     max_context_len, sm_scale, out, lse=None, workspace=None, cos_sin=None,
                     window=-1, chunk_blocks=0, k_scale=None, v_scale=None, sinks=None, stream=None):
    """pkv_decode_step with every argument marshalled once (see BoundCall)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    max_pos = 0 if cos_sin is None else int(cos_sin.shape[0])
    desc_copy = CacheDesc.from_buffer_copy(desc)
    args = (ctypes.byref(desc_copy), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(cos_sin), max_pos,
            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
            _ptr(context_lens), int(context_lens.shape[0]), int(max_context_len), float(sm_scale),
            int(window), _ptr(sinks), int(chunk_blocks), _ptr(out), _ptr(lse), _ptr(workspace),
            ws_bytes, _stream(stream))
    keep = (desc_copy, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, lse,
            workspace, cos_sin, k_scale, v_scale, sinks)
    return BoundCall(load_library().pkv_decode_step, args, keep)


def pkv_decode_attention_static(desc, q, k_cache, v_cache, block_tables, context_lens,
                                max_context_len, sm_scale, out, lse=None, window=-1,
                                chunk_blocks=0, k_scale=None, v_scale=None, sinks=None,
                                stream=None):
    """Decode for callers that cannot allocate: no workspace argument, the
    library's fixed 16 MiB device scratch instead (see include/pkv.h)."""
    _check(load_library().pkv_decode_attention_static(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(context_lens), int(context_lens.shape[0]), int(max_context_len),
        float(sm_scale), int(window), _ptr(sinks), int(chunk_blocks), _ptr(out), _ptr(lse),
        _stream(stream)))


def pkv_prefill_workspace_size(desc, num_seqs, total_q_tokens) -> int:
    return int(load_library().pkv_prefill_workspace_size(ctypes.byref(desc), int(num_seqs),
                                                         int(total_q_tokens)))


def pkv_prefill_attention_ragged(desc, q, qo_indptr, k_cache, v_cache, block_tables, kv_lens,
                                 sm_scale, out, lse=None, qo_indptr_host=None, kv_lens_host=None,
                                 causal=True, window=-1, workspace=None, k_scale=None,
                                 v_scale=None, stream=None):
    qh = None if qo_indptr_host is None else np.ascontiguousarray(qo_indptr_host, np.int32)
    kh = None if kv_lens_host is None else np.ascontiguousarray(kv_lens_host, np.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().pkv_prefill_attention_ragged(
        ctypes.byref(desc), _ptr(q), _ptr(qo_indptr), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(kv_lens), int(kv_lens.shape[0]),
        int(q.shape[0]), _ptr(qh), _ptr(kh), float(sm_scale), int(bool(causal)), int(window),
        _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_prefill_ring_workspace_size(desc, num_seqs, window, max_q_len):
    return int(load_library().pkv_prefill_ring_workspace_size(ctypes.byref(desc), int(num_seqs),
                                                              int(window), int(max_q_len)))


def pkv_prefill_ring_commit(desc, q, qo_indptr, k_chunk, v_chunk, k_cache, v_cache, block_tables,
                            kv_lens, sm_scale, window, out, qo_indptr_host, kv_lens_host,
                            workspace, lse=None, k_scale=None, v_scale=None, stream=None):
    """Ragged prefill over a ring cache, then the commit of the chunk's K/V
    (k_chunk / v_chunk, bf16 [total_q][Hkv][D], K after RoPE) into the ring."""
    qh = np.ascontiguousarray(qo_indptr_host, np.int32)
    kh = np.ascontiguousarray(kv_lens_host, np.int32)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().pkv_prefill_ring_commit(
        ctypes.byref(desc), _ptr(q), _ptr(qo_indptr), _ptr(k_chunk), _ptr(v_chunk), _ptr(k_cache),
        _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(kv_lens),
        int(kv_lens.shape[0]), int(q.shape[0]), _ptr(qh), _ptr(kh), float(sm_scale), int(window),
        _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def pkv_merge_states(o_parts, lse_parts, out, lse_out=None, stream=None):
    """o_parts fp32 [P][rows][H][D], lse_parts fp32 [P][rows][H] -> out bf16 [rows][H][D]."""
    P, rows, H, D = o_parts.shape
    _check(load_library().pkv_merge_states(_ptr(o_parts), _ptr(lse_parts), int(P), int(rows),
                                           int(H), int(D), _ptr(out), _ptr(lse_out),
                                           _stream(stream)))


def pkv_cascade_workspace_size(desc, num_groups, num_seqs, max_prefix_len, max_suffix_len,
                               window=-1):
    return int(load_library().pkv_cascade_workspace_size(
        ctypes.byref(desc), int(num_groups), int(num_seqs), int(max_prefix_len),
        int(max_suffix_len), int(window)))


def pkv_cascade_decode(desc, q, k_cache, v_cache, group_indptr, group_indptr_host, prefix_tables,
                       prefix_lens, prefix_lens_host, suffix_tables, suffix_lens, max_suffix_len,
                       sm_scale, out, lse=None, workspace=None, window=-1, k_scale=None,
                       v_scale=None, stream=None):
    gh = np.ascontiguousarray(group_indptr_host, np.int32)
    ph = np.ascontiguousarray(prefix_lens_host, np.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().pkv_cascade_decode(
        ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        int(gh.shape[0] - 1), _ptr(group_indptr), _ptr(gh), _ptr(prefix_tables), _ptr(prefix_lens),
        _ptr(ph), int(q.shape[0]), _ptr(suffix_tables), _ptr(suffix_lens), int(max_suffix_len),
        float(sm_scale), int(window), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        _stream(stream)))


def pkv_device_errors(reset: bool = True) -> int:
    """Synchronously read (and by default clear) the device error word."""
    v = ctypes.c_uint32()
    _check(load_library().pkv_device_errors(ctypes.byref(v), int(bool(reset))))
    return int(v.value)


def pkv_test_inject_wait_timeout(kernels: int, limit_us: int = 0) -> None:
    """Testing only: arm (kernels bit 0 decode, bit 1 tcgen05 prefill) or
    disarm (0) the library's give-up path of one bounded wait per launch."""
    _check(load_library().pkv_test_inject_wait_timeout(int(kernels), int(limit_us)))


def pkv_last_error() -> str:
    return load_library().pkv_last_error().decode(errors="replace")


__all__ = [n for n in dir() if n.startswith("pkv_")] + [
    "CacheDesc", "make_desc", "PkvError", "load_library", "library_path", "KV_BF16",
    "KV_FP8_E4M3", "BoundCall", "bind_decode_step"]
