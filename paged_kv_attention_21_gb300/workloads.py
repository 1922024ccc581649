"""Seeded synthetic inputs for attention over a paged KV cache.

This module draws numbers and lays them out -- sequence lengths, block
tables, pool contents, queries -- and holds none of the attention, RoPE or
merge arithmetic.  Tests and ``bench.py`` feed what it returns, byte for byte,
to both the CUDA library and the CPU oracle.

Recipe (shared by every workload):

* lengths and block tables come from ``numpy.random.default_rng(seed)``;
  physical blocks are drawn without replacement from the pool, so tables are
  scattered over it (the paged cache of PagedAttention: infer-lab "Technique"
  table, llm-infer "What It Does");
* every pool element, used or not, and every query is N(0, 1) from a
  ``torch.Generator`` seeded with the same seed, rounded to bf16 by torch;
* an e4m3 pool keeps one fp32 scale per KV head, frozen from a warm-up slice
  of the data as amax / 448 (InferX, "The kernels underneath": per-layer K/V
  scales freeze from warmup); the codes are torch's float8_e4m3fn cast of
  value / scale, so later values beyond the warm-up range saturate;
* table entries past a sequence's last block are -1.

The five workloads are shaped like the layers the pages serve (Qwen2.5-3B,
Qwen3-4B, Llama-3-8B), with block_size 16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    """One decode batch: B sequences, one query token each."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx_lo: int
    ctx_hi: int
    seed: int
    kv_dtype: str = "bf16"            # "bf16" or "fp8_e4m3"
    pool_blocks: Optional[int] = None  # None: 1.5x the blocks the batch needs
    fixed_lens: Optional[tuple] = None
    rope_theta: float = 1.0e6          # used when the new token is appended
    block_size: int = BLOCK_SIZE

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclasses.dataclass(frozen=True)
class PrefillSpec:
    """Ragged causal chunked prefill: pairs of sequences share a cached prefix."""

    name: str
    num_chunks: int
    chunk_len: int
    prefix_lo: int
    prefix_hi: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int
    block_size: int = BLOCK_SIZE

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclasses.dataclass(frozen=True)
class CascadeSpec:
    """Groups of decode sequences sharing a block-aligned cached prefix (a
    radix-cache hit), each with its own suffix."""

    name: str
    groups: int
    group_size: int
    prefix_lo: int
    prefix_hi: int
    suffix_lo: int
    suffix_hi: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int
    block_size: int = BLOCK_SIZE

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads.  Names say what they are shaped like.
TINY = DecodeSpec("tiny decode, 4 seqs, 8/2 heads, D64", batch=4, num_q_heads=8, num_kv_heads=2,
                  head_dim=64, ctx_lo=17, ctx_hi=255, seed=20261, pool_blocks=64,
                  fixed_lens=(17, 64, 100, 255))
QWEN25_3B = DecodeSpec("Qwen2.5-3B-shaped decode, B64, 16/2 heads, D128, ctx 256-4096",
                       batch=64, num_q_heads=16, num_kv_heads=2, head_dim=128, ctx_lo=256,
                       ctx_hi=4096, seed=20262, pool_blocks=40000)
QWEN3_4B = DecodeSpec("Qwen3-4B-shaped decode + append, B256, 32/8 heads, D128, ctx 256-768",
                      batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128, ctx_lo=256,
                      ctx_hi=768, seed=20263)
LLAMA3_8B_DECODE = DecodeSpec("Llama-3-8B-shaped mixed step, decode part, B120, ctx 1024-32768",
                              batch=120, num_q_heads=32, num_kv_heads=8, head_dim=128,
                              ctx_lo=1024, ctx_hi=32768, seed=20264)
LLAMA3_8B_PREFILL = PrefillSpec("Llama-3-8B-shaped mixed step, prefill part, 8x512 over 0-8192",
                                num_chunks=8, chunk_len=512, prefix_lo=0, prefix_hi=8192,
                                num_q_heads=32, num_kv_heads=8, head_dim=128, seed=20264)
FP8_DECODE = DecodeSpec("FP8 e4m3 decode, B128, 64/8 heads, D64, ctx 1024-16384",
                        batch=128, num_q_heads=64, num_kv_heads=8, head_dim=64, ctx_lo=1024,
                        ctx_hi=16384, seed=20265, kv_dtype="fp8_e4m3")
FP8_WINDOW = 128  # the sliding-window layer of the FP8 workload
FP8_RING = 9      # ring blocks that hold any 128-key window: ceil((128 - 1) / 16) + 1

# Supplementary workloads of the next-step rows (not the headline).
CASCADE_DECODE = CascadeSpec("shared-prefix decode: 16 groups x 8 sequences, prefix U[1024,8192] "
                             "(block-aligned), suffix U[16,512], 32/8 heads, D128",
                             groups=16, group_size=8, prefix_lo=1024, prefix_hi=8192, suffix_lo=16,
                             suffix_hi=512, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=20266)
VERIFY_Q_LENS = (2, 8)  # speculative-verify query tokens per sequence, uniform

CONFIGS = {1: TINY, 2: QWEN25_3B, 3: QWEN3_4B, 4: LLAMA3_8B_DECODE, 5: FP8_DECODE}


def scaled(spec: DecodeSpec, batch: int, ctx_hi: Optional[int] = None, pool_blocks=None,
           seed: Optional[int] = None) -> DecodeSpec:
    """The same shape with fewer sequences / shorter contexts (parity sizes)."""
    hi = spec.ctx_hi if ctx_hi is None else ctx_hi
    return dataclasses.replace(spec, batch=batch, ctx_hi=hi, ctx_lo=min(spec.ctx_lo, hi),
                               pool_blocks=pool_blocks, fixed_lens=None,
                               seed=spec.seed if seed is None else seed)


# ------------------------------------------------------------- primitives --

def draw_lengths(spec: DecodeSpec, rng: np.random.Generator) -> np.ndarray:
    if spec.fixed_lens is not None:
        return np.asarray(spec.fixed_lens, dtype=np.int32)
    return rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=spec.batch).astype(np.int32)


def blocks_for(lens, block_size=BLOCK_SIZE) -> np.ndarray:
    return (np.asarray(lens, dtype=np.int64) + block_size - 1) // block_size


def allocate_tables(lens, free_blocks: np.ndarray, rng: np.random.Generator,
                    block_size=BLOCK_SIZE, max_blocks_per_seq=None):
    """Give each sequence its own blocks, drawn without replacement from
    ``free_blocks`` in random order.  Returns (tables [B][mbps] int32 with -1
    past each sequence's last block, the blocks left over)."""
    nblk = blocks_for(lens, block_size)
    need = int(nblk.sum())
    if need > len(free_blocks):
        raise ValueError("pool too small: need %d blocks, have %d" % (need, len(free_blocks)))
    order = rng.permutation(len(free_blocks))
    picked = free_blocks[order[:need]]
    rest = free_blocks[order[need:]]
    mbps = int(max(1, nblk.max() if len(nblk) else 1)) if max_blocks_per_seq is None \
        else max_blocks_per_seq
    tables = np.full((len(nblk), mbps), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = picked[off:off + n]
        off += n
    return tables, rest


def _normal(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def fill_bf16(shape, gen: torch.Generator, device, chunk_rows: int = 4096) -> torch.Tensor:
    """N(0,1) rounded to bf16, generated in slices of the leading dim."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        out[a:b] = _normal((b - a,) + tuple(shape[1:]), gen, device).to(torch.bfloat16)
    return out


def fill_e4m3(shape, gen: torch.Generator, device, chunk_rows: int = 4096):
    """N(0,1) quantised to e4m3 codes (uint8) with one scale per dim-1 index
    (the KV head), frozen from the first slice.  Returns (codes, scales)."""
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    scales = None
    for a in range(0, shape[0], chunk_rows):
        b = min(shape[0], a + chunk_rows)
        x = _normal((b - a,) + tuple(shape[1:]), gen, device)
        if scales is None:
            amax = x.abs().transpose(0, 1).reshape(shape[1], -1).amax(dim=1)
            scales = (amax / 448.0).to(torch.float32)
        bshape = (1, shape[1]) + (1,) * (len(shape) - 2)
        y = (x / scales.view(bshape)).clamp(-448.0, 448.0)
        out[a:b] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return out, scales


# --------------------------------------------------------------- batches --

@dataclasses.dataclass
class DecodeBatch:
    spec: DecodeSpec
    q: torch.Tensor              # bf16 [B][Hq][D]
    k_cache: torch.Tensor        # bf16 or uint8 [NB][Hkv][bs][D]
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]  # fp32 [Hkv] (e4m3 only)
    v_scale: Optional[torch.Tensor]
    block_tables: torch.Tensor   # int32 [B][mbps]
    context_lens: torch.Tensor   # int32 [B]
    k_new: torch.Tensor          # bf16 [B][Hkv][D]: the token appended at ctx-1
    v_new: torch.Tensor
    lens_host: np.ndarray
    tables_host: np.ndarray

    @property
    def max_context_len(self) -> int:
        return int(self.lens_host.max()) if len(self.lens_host) else 0

    def kv_bytes(self, window: int = -1) -> int:
        """Algorithmic K+V bytes one decode pass reads (visible keys only)."""
        s = self.spec
        elem = 1 if s.kv_dtype == "fp8_e4m3" else 2
        vis = self.lens_host.astype(np.int64)
        if window > 0:
            vis = np.minimum(vis, window)
        return int(vis.sum()) * s.num_kv_heads * s.head_dim * elem * 2


def make_decode_batch(spec: DecodeSpec, device="cpu", pool=None, free_blocks=None,
                      seed_offset: int = 0, max_blocks_per_seq=None) -> DecodeBatch:
    """Draw one decode batch.  With ``pool=(k_cache, v_cache, k_scale,
    v_scale)`` and ``free_blocks`` the batch takes its blocks from an existing
    pool (several batches over disjoint regions of one pool)."""
    seed = spec.seed + seed_offset
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device).manual_seed(seed)
    lens = draw_lengths(spec, rng)
    bs = spec.block_size
    if pool is None:
        need = int(blocks_for(lens, bs).sum())
        nb = spec.pool_blocks if spec.pool_blocks is not None else max(need, int(need * 1.5))
        shape = (nb, spec.num_kv_heads, bs, spec.head_dim)
        if spec.kv_dtype == "fp8_e4m3":
            k_cache, k_scale = fill_e4m3(shape, gen, device)
            v_cache, v_scale = fill_e4m3(shape, gen, device)
        else:
            k_cache, k_scale = fill_bf16(shape, gen, device), None
            v_cache, v_scale = fill_bf16(shape, gen, device), None
        free_blocks = np.arange(nb, dtype=np.int32)
    else:
        k_cache, v_cache, k_scale, v_scale = pool
    if spec.fixed_lens is not None and free_blocks is not None and len(free_blocks) == \
            k_cache.shape[0]:
        # the tiny workload: a random permutation of the whole pool, in order
        perm = rng.permutation(k_cache.shape[0]).astype(np.int32)
        nblk = blocks_for(lens, bs)
        mbps = int(nblk.max())
        tables = np.full((len(lens), mbps), -1, dtype=np.int32)
        off = 0
        for s, n in enumerate(nblk):
            tables[s, :n] = perm[off:off + n]
            off += n
    else:
        tables, _ = allocate_tables(lens, np.asarray(free_blocks), rng, bs, max_blocks_per_seq)
    q = fill_bf16((spec.batch, spec.num_q_heads, spec.head_dim), gen, device)
    k_new = fill_bf16((spec.batch, spec.num_kv_heads, spec.head_dim), gen, device)
    v_new = fill_bf16((spec.batch, spec.num_kv_heads, spec.head_dim), gen, device)
    return DecodeBatch(spec=spec, q=q, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
                       v_scale=v_scale, block_tables=torch.from_numpy(tables).to(device),
                       context_lens=torch.from_numpy(lens).to(device), k_new=k_new, v_new=v_new,
                       lens_host=lens, tables_host=tables)


def make_decode_instances(spec: DecodeSpec, n: int, device="cpu"):
    """``n`` decode batches of one shape over disjoint regions of one pool
    (each instance draws its own lengths, tables and queries); every table
    has ceil(ctx_hi / block_size) columns."""
    mbps = (spec.ctx_hi + spec.block_size - 1) // spec.block_size
    if spec.pool_blocks is None and n > 1:
        # room for n batches at the longest lengths, plus slack
        spec = dataclasses.replace(spec, pool_blocks=int(1.25 * n * spec.batch * mbps) + 16)
    first = make_decode_batch(spec, device, max_blocks_per_seq=mbps)
    pool = (first.k_cache, first.v_cache, first.k_scale, first.v_scale)
    used = set(first.tables_host[first.tables_host >= 0].tolist())
    out = [first]
    for i in range(1, n):
        free = np.array([b for b in range(first.k_cache.shape[0]) if b not in used],
                        dtype=np.int32)
        inst = make_decode_batch(spec, device, pool=pool, free_blocks=free, seed_offset=1000 * i,
                                 max_blocks_per_seq=mbps)
        used |= set(inst.tables_host[inst.tables_host >= 0].tolist())
        out.append(inst)
    return out


@dataclasses.dataclass
class PrefillBatch:
    spec: PrefillSpec
    q: torch.Tensor              # bf16 [sum q][Hq][D]
    k_cache: torch.Tensor        # bf16 [NB][Hkv][bs][D], chunk K/V already in place
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [B][mbps]
    qo_indptr: torch.Tensor      # int32 [B+1]
    kv_lens: torch.Tensor        # int32 [B]
    qo_indptr_host: np.ndarray
    kv_lens_host: np.ndarray
    tables_host: np.ndarray
    prefix_host: np.ndarray      # cached prefix length per sequence

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr_host[-1])

    def flops(self) -> int:
        """Algorithmic causal flops: 4*D*Hq * sum_s (q*prefix + q(q+1)/2)."""
        s = self.spec
        q = np.diff(self.qo_indptr_host).astype(np.int64)
        p = self.prefix_host.astype(np.int64)
        return int(4 * s.head_dim * s.num_q_heads * np.sum(q * p + q * (q + 1) // 2))


def make_prefill_batch(spec: PrefillSpec, device="cpu", pool=None, free_blocks=None,
                       q_lens=None, prefixes=None) -> PrefillBatch:
    """Pairs of sequences share a cached prefix: the prefix's full blocks
    appear in both tables (same physical ids); a partial last prefix block is
    copied per sequence with identical bytes; each sequence then owns the
    blocks of its new chunk.  ``q_lens`` / ``prefixes`` override the draw."""
    rng = np.random.default_rng(spec.seed + 7)
    gen = torch.Generator(device=device).manual_seed(spec.seed + 7)
    bs = spec.block_size
    B = spec.num_chunks
    if prefixes is None:
        npairs = (B + 1) // 2
        pair_prefix = rng.integers(spec.prefix_lo, spec.prefix_hi + 1, size=npairs)
        prefixes = np.repeat(pair_prefix, 2)[:B].astype(np.int32)
    prefixes = np.asarray(prefixes, dtype=np.int32)
    q_lens = np.full(B, spec.chunk_len, dtype=np.int32) if q_lens is None \
        else np.asarray(q_lens, dtype=np.int32)
    kv_lens = (prefixes + q_lens).astype(np.int32)
    shared = prefixes // bs                       # full prefix blocks, shared by a pair
    own = blocks_for(kv_lens, bs) - shared        # tail copy + chunk blocks
    npairs = (B + 1) // 2
    need = int(sum(shared[2 * j] for j in range(npairs)) + own.sum())
    if pool is None:
        nb = max(need, int(need * 1.25))
        shape = (nb, spec.num_kv_heads, bs, spec.head_dim)
        k_cache = fill_bf16(shape, gen, device)
        v_cache = fill_bf16(shape, gen, device)
        free_blocks = np.arange(nb, dtype=np.int32)
    else:
        k_cache, v_cache = pool
    free = np.asarray(free_blocks)[rng.permutation(len(free_blocks))]
    mbps = int(blocks_for(kv_lens, bs).max())
    tables = np.full((B, mbps), -1, dtype=np.int32)
    off = 0
    for j in range(npairs):
        ids = free[off:off + shared[2 * j]]
        off += shared[2 * j]
        for s in (2 * j, 2 * j + 1):
            if s >= B:
                continue
            tables[s, :shared[s]] = ids
            tables[s, shared[s]:shared[s] + own[s]] = free[off:off + own[s]]
            off += own[s]
        a, b = 2 * j, 2 * j + 1
        r = prefixes[a] % bs
        if b < B and r:
            # identical bytes for the copied partial prefix block
            ta, tb = int(tables[a, shared[a]]), int(tables[b, shared[b]])
            k_cache[tb, :, :r] = k_cache[ta, :, :r]
            v_cache[tb, :, :r] = v_cache[ta, :, :r]
    qo = np.zeros(B + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    q = fill_bf16((int(qo[-1]), spec.num_q_heads, spec.head_dim), gen, device)
    return PrefillBatch(spec=spec, q=q, k_cache=k_cache, v_cache=v_cache,
                        block_tables=torch.from_numpy(tables).to(device),
                        qo_indptr=torch.from_numpy(qo).to(device),
                        kv_lens=torch.from_numpy(kv_lens).to(device), qo_indptr_host=qo,
                        kv_lens_host=kv_lens, tables_host=tables, prefix_host=prefixes)


@dataclasses.dataclass
class CascadeBatch:
    spec: CascadeSpec
    q: torch.Tensor                # bf16 [B][Hq][D]
    k_cache: torch.Tensor          # bf16 [NB][Hkv][bs][D]
    v_cache: torch.Tensor
    group_indptr: torch.Tensor     # int32 [groups + 1]
    prefix_tables: torch.Tensor    # int32 [groups][mbps]
    prefix_lens: torch.Tensor      # int32 [groups]
    suffix_tables: torch.Tensor    # int32 [B][mbps]
    suffix_lens: torch.Tensor      # int32 [B]
    concat_tables: torch.Tensor    # int32 [B][mbps]: prefix blocks then suffix blocks
    concat_lens: torch.Tensor      # int32 [B]
    group_indptr_host: np.ndarray
    prefix_host: np.ndarray
    suffix_host: np.ndarray

    def cascade_kv_bytes(self) -> int:
        """K+V bytes with each group's prefix read once."""
        s = self.spec
        toks = int(self.prefix_host.astype(np.int64).sum() + self.suffix_host.astype(np.int64).sum())
        return toks * s.num_kv_heads * s.head_dim * 2 * 2

    def uncached_kv_bytes(self) -> int:
        """K+V bytes of plain decode over each sequence's whole context."""
        s = self.spec
        per_seq = np.repeat(self.prefix_host, s.group_size).astype(np.int64) + self.suffix_host
        return int(per_seq.sum()) * s.num_kv_heads * s.head_dim * 2 * 2


def make_cascade_batch(spec: CascadeSpec, device="cpu") -> CascadeBatch:
    """Seeded shared-prefix batch: group g's prefix blocks are shared by its
    sequences (one table row per group); each sequence's suffix has its own
    blocks.  Prefixes are whole blocks, so the concatenated table of a
    sequence is its prefix blocks followed by its suffix blocks."""
    rng = np.random.default_rng(spec.seed)
    gen = torch.Generator(device=device).manual_seed(spec.seed)
    bs = spec.block_size
    B = spec.groups * spec.group_size
    prefix = (bs * rng.integers(spec.prefix_lo // bs, spec.prefix_hi // bs + 1,
                                size=spec.groups)).astype(np.int32)
    suffix = rng.integers(spec.suffix_lo, spec.suffix_hi + 1, size=B).astype(np.int32)
    pblk = prefix // bs
    sblk = blocks_for(suffix, bs)
    need = int(pblk.sum() + sblk.sum())
    nb = int(need * 1.25) + 16
    shape = (nb, spec.num_kv_heads, bs, spec.head_dim)
    k_cache = fill_bf16(shape, gen, device)
    v_cache = fill_bf16(shape, gen, device)
    ids = rng.permutation(nb).astype(np.int32)
    mbps = int(pblk.max() + sblk.max())
    ptab = np.full((spec.groups, mbps), -1, np.int32)
    stab = np.full((B, mbps), -1, np.int32)
    ctab = np.full((B, mbps), -1, np.int32)
    off = 0
    for g in range(spec.groups):
        ptab[g, :pblk[g]] = ids[off:off + pblk[g]]
        off += pblk[g]
    for i in range(B):
        g = i // spec.group_size
        stab[i, :sblk[i]] = ids[off:off + sblk[i]]
        off += sblk[i]
        ctab[i, :pblk[g]] = ptab[g, :pblk[g]]
        ctab[i, pblk[g]:pblk[g] + sblk[i]] = stab[i, :sblk[i]]
    gptr = (spec.group_size * np.arange(spec.groups + 1)).astype(np.int32)
    q = fill_bf16((B, spec.num_q_heads, spec.head_dim), gen, device)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return CascadeBatch(spec=spec, q=q, k_cache=k_cache, v_cache=v_cache, group_indptr=t(gptr),
                        prefix_tables=t(ptab), prefix_lens=t(prefix), suffix_tables=t(stab),
                        suffix_lens=t(suffix), concat_tables=t(ctab),
                        concat_lens=t(np.repeat(prefix, spec.group_size) + suffix),
                        group_indptr_host=gptr, prefix_host=prefix, suffix_host=suffix)
