"""Plain CPU oracle for attention over a paged KV cache -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu_baseline leg (and the
``--impl reference`` arm) of ``bench.py`` may import this package.  The CUDA
library never loads it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp32 with an fp64 variant,
built with ``-ffp-contract=off`` so every product and sum is rounded on its
own).  This module only compiles it with gcc and marshals numpy arrays.

Function by function, what each follows (the page title, then the section):

* ``bf16_from_f32`` / ``f32_from_bf16`` -- bf16 storage of the cache
  (InferX, "Against vLLM": bf16 serving); RNE narrowing.
* ``e4m3_from_f32`` / ``f32_from_e4m3`` -- FP8 e4m3 KV cache (InferX, "The
  kernels underneath", M8 FP8 KV cache); OCP E4M3FN, RNE, saturating.
* ``rope_table`` / ``append_rope`` -- the KV write fused with RoPE (llm-infer,
  "What It Does"; infer-lab source layout: RoPE, GQA).
* ``gather_kv`` -- block-table addressing (infer-lab, "Technique" table:
  PagedAttention block tables).
* ``copy_blocks`` -- copy-on-write of shared blocks (infer-lab, "Technique"
  table: refcounting, copy-on-write; llm-infer, "What It Does").
* ``paged_attention`` -- softmax attention over the paged cache: decode,
  ragged causal chunked prefill, sliding window (infer-lab invariants;
  llm-infer "References": FlashAttention-2; RustInfer "Status": 128-token SWA).
* ``merge_states`` -- merge of partial (o, lse) states (FlashAttention-2 work
  partitioning, llm-infer "References").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpkv_oracle.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/libpkv_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f32.restype = f32
        lib.orc_f32_to_bf16.argtypes = [f32]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f32.restype = f32
        lib.orc_f32_to_e4m3.argtypes = [f32]
        lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
        lib.orc_rope_table.argtypes = [f32, i32, i32, P]
        lib.orc_rope_table.restype = None
        lib.orc_append_rope.argtypes = [i32, i32, i32, i32, i32, i64, i32, i32, P, P, P, P, P,
                                        i32, P, P, i32, P, P, P, P, i32]
        lib.orc_append_rope.restype = ctypes.c_int
        lib.orc_gather_kv.argtypes = [i32, i32, i32, i32, i64, i32, P, P, P, i32, P]
        lib.orc_gather_kv.restype = ctypes.c_int
        lib.orc_paged_attention.argtypes = [i32, i32, i32, i32, i32, i64, i32, P, P, P, P, P,
                                            i32, P, P, P, f32, i32, i32, i32, P, P, P, i32, i32]
        lib.orc_paged_attention.restype = ctypes.c_int
        lib.orc_copy_blocks.argtypes = [P, i64, i64, P, P, i32]
        lib.orc_copy_blocks.restype = ctypes.c_int
        lib.orc_merge_states.argtypes = [P, P, i32, i32, i32, i32, P, P]
        lib.orc_merge_states.restype = None
        for name in ("orc_bf16_to_f32_array", "orc_f32_to_bf16_array", "orc_e4m3_to_f32_array",
                     "orc_f32_to_e4m3_array"):
            getattr(lib, name).argtypes = [P, P, i64]
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------- conversions --

def _convert(fn_name, x, in_dtype, out_dtype):
    x = _c(x, in_dtype)
    out = np.empty(x.shape, dtype=out_dtype)
    getattr(_load(), fn_name)(_ptr(x), _ptr(out), x.size)
    return out


def f32_from_bf16(bits):
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return _convert("orc_bf16_to_f32_array", bits, np.uint16, np.float32)


def bf16_from_f32(x):
    """float32 -> bf16 bit patterns, round to nearest even."""
    return _convert("orc_f32_to_bf16_array", x, np.float32, np.uint16)


def f32_from_e4m3(codes):
    """e4m3 codes (uint8) -> float32 (exact)."""
    return _convert("orc_e4m3_to_f32_array", codes, np.uint8, np.float32)


def e4m3_from_f32(x):
    """float32 -> e4m3 codes, round to nearest even, saturating to +-448."""
    return _convert("orc_f32_to_e4m3_array", x, np.float32, np.uint8)


# ------------------------------------------------------------------ RoPE --

def rope_table(theta: float, rotary_dim: int, max_pos: int) -> np.ndarray:
    """fp32 [max_pos][rotary_dim/2][2] table of (cos, sin)."""
    lib = _load()
    out = np.empty((max_pos, rotary_dim // 2, 2), dtype=np.float32)
    lib.orc_rope_table(float(theta), int(rotary_dim), int(max_pos), _ptr(out))
    return out


def append_rope(*, num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype, k_cache, v_cache,
                block_tables, token_to_seq, positions, k_new, v_new, q=None, cos_sin=None,
                k_scale=None, v_scale=None, ring_blocks=0):
    """Host append + RoPE.  Mutates k_cache / v_cache (numpy, uint16 for bf16
    or uint8 for e4m3, shape [num_blocks][Hkv][bs][D]) and returns the rotated
    q (a new uint16 array) or None."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    bt = _c(block_tables, np.int32)
    num_seqs, mbps = bt.shape
    tts = _c(token_to_seq, np.int32)
    pos = _c(positions, np.int32)
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    qo = None if q is None else np.array(q, dtype=np.uint16, copy=True, order="C")
    cs = None if cos_sin is None else _c(cos_sin, np.float32)
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    max_pos = 0 if cs is None else cs.shape[0]
    rc = lib.orc_append_rope(num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                             k_cache.shape[0], mbps, int(ring_blocks), _ptr(k_cache), _ptr(v_cache), _ptr(ks),
                             _ptr(vs), _ptr(bt), num_seqs, _ptr(tts), _ptr(pos), len(pos),
                             _ptr(kn), _ptr(vn), _ptr(qo), _ptr(cs), max_pos)
    if rc != 0:
        raise ValueError("oracle append_rope: out-of-range index (rc=%d)" % rc)
    return qo


def copy_blocks(cache, src, dst):
    """Copy-on-write: block dst[i] of the pool (numpy, mutated) gets block src[i]."""
    lib = _load()
    assert cache.flags.c_contiguous
    s = _c(src, np.int32)
    d = _c(dst, np.int32)
    block_bytes = cache[0].nbytes
    rc = lib.orc_copy_blocks(_ptr(cache), cache.shape[0], block_bytes, _ptr(s), _ptr(d), len(s))
    if rc != 0:
        raise ValueError("oracle copy_blocks: out-of-range block id")


def gather_kv(cache, block_tables, lens, *, block_size):
    """Paged -> contiguous [sum(lens)][Hkv][D] copy of one pool."""
    lib = _load()
    cache = np.ascontiguousarray(cache)
    nb, hkv, bs, d = cache.shape
    assert bs == block_size
    bt = _c(block_tables, np.int32)
    ln = _c(lens, np.int32)
    out = np.empty((int(ln.sum()), hkv, d), dtype=cache.dtype)
    rc = lib.orc_gather_kv(hkv, d, bs, cache.dtype.itemsize, nb, bt.shape[1], _ptr(cache),
                           _ptr(bt), _ptr(ln), len(ln), _ptr(out))
    if rc != 0:
        raise ValueError("oracle gather_kv: out-of-range index")
    return out


def paged_attention(*, q, k_cache, v_cache, block_tables, qo_indptr, kv_lens, num_q_heads,
                    num_kv_heads, sm_scale, causal=True, window=-1, kv_dtype=KV_BF16,
                    k_scale=None, v_scale=None, precision=32, nthreads=1, with_lse=True,
                    ring_blocks=0, sinks=None):
    """Ragged softmax attention over the paged cache.

    q: uint16 bf16 bits [T][Hq][D].  Returns (out fp32 [T][Hq][D], lse fp32
    [T][Hq]).  Decode is qo_indptr = arange(B + 1)."""
    lib = _load()
    q = _c(q, np.uint16)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    nb, hkv, bs, d = k_cache.shape
    assert hkv == num_kv_heads
    bt = _c(block_tables, np.int32)
    qo = _c(qo_indptr, np.int32)
    kl = _c(kv_lens, np.int32)
    T = int(qo[-1])
    out = np.empty((T, num_q_heads, d), dtype=np.float32)
    lse = np.empty((T, num_q_heads), dtype=np.float32) if with_lse else None
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    rc = lib.orc_paged_attention(num_q_heads, hkv, d, bs, kv_dtype, nb, bt.shape[1],
                                 _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs), _ptr(bt),
                                 len(kl), _ptr(qo), _ptr(kl), _ptr(q), float(sm_scale),
                                 int(causal), int(window), int(ring_blocks),
                                 _ptr(None if sinks is None else _c(sinks, np.float32)),
                                 _ptr(out), _ptr(lse), int(precision),
                                 int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged_attention failed (rc=%d)" % rc)
    return out, lse


def merge_states(o_parts, lse_parts):
    """o_parts fp32 [P][rows][H][D], lse_parts [P][rows][H] -> (o, lse)."""
    lib = _load()
    o_parts = _c(o_parts, np.float32)
    lse_parts = _c(lse_parts, np.float32)
    P, rows, H, D = o_parts.shape
    out = np.empty((rows, H, D), dtype=np.float32)
    lse = np.empty((rows, H), dtype=np.float32)
    lib.orc_merge_states(_ptr(o_parts), _ptr(lse_parts), P, rows, H, D, _ptr(out), _ptr(lse))
    return out, lse
