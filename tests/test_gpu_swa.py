"""GPU parity of the sliding-window layer's cache and softmax (RustInfer,
"Status": SWA with a 128-token ring cache and attention sinks): decode over a
ring of blocks per sequence, append into the ring, and per-head sink logits --
each against the oracle element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from tests._cases import BS, PagedCase, bf16_bits
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _dev_pool(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if bits.dtype == np.uint16:
        return t.view(torch.int16).view(torch.bfloat16).to(DEV)
    return t.to(DEV)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _ring_from_linear(case, ring):
    """Ring entry b % ring of each sequence holds the last logical block b
    that maps there (numpy copies)."""
    B = len(case.lens)
    k = np.zeros((B * ring,) + case.k_cache.shape[1:], case.k_cache.dtype)
    v = np.zeros_like(k)
    tabs = (np.arange(ring)[None, :] + ring * np.arange(B)[:, None]).astype(np.int32)
    for s in range(B):
        for b in range((int(case.lens[s]) + BS - 1) // BS):
            k[tabs[s, b % ring]] = case.k_cache[case.tables[s, b]]
            v[tabs[s, b % ring]] = case.v_cache[case.tables[s, b]]
    return k, v, tabs


def _decode(case, k, v, tabs, window, ring=0, sinks=None, chunk=0, static=False):
    desc = pkv.make_desc(num_q_heads=case.hq, num_kv_heads=case.hkv, head_dim=case.d,
                         num_blocks=k.shape[0], max_blocks_per_seq=tabs.shape[1],
                         kv_dtype=1 if case.fp8 else 0, ring_blocks=ring)
    B = len(case.lens)
    max_ctx = int(case.lens.max())
    q = _dev_pool(case.q)
    out = torch.full((B, case.hq, case.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, case.hq), float("nan"), device=DEV)
    ks = None if case.k_scale is None else _dev(case.k_scale)
    vs = None if case.v_scale is None else _dev(case.v_scale)
    sk = None if sinks is None else _dev(sinks)
    args = (desc, q, _dev_pool(k), _dev_pool(v), _dev(tabs), _dev(case.lens), max_ctx, 1 / math.sqrt(case.d),
            out, lse)
    if static:
        pkv.pkv_decode_attention_static(*args, window=window, chunk_blocks=chunk, k_scale=ks, v_scale=vs,
                                        sinks=sk)
    else:
        size = pkv.pkv_decode_workspace_size(desc, B, max_ctx, window, chunk)
        ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=DEV)
        pkv.pkv_decode_attention(*args, workspace=ws, window=window, chunk_blocks=chunk, k_scale=ks,
                                 v_scale=vs, sinks=sk)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("fp8", [False, True])
def test_ring_decode_matches_oracle_and_linear_cache(fp8):
    rng = np.random.default_rng(50 + fp8)
    hq, hkv, d = (64, 8, 64) if fp8 else (32, 8, 128)
    lens = [1, 15, 16, 17, 128, 129, 144, 145, 700, 3001, 16384]
    case = PagedCase(rng, lens, hq, hkv, d, fp8=fp8)
    window, ring = 128, 9
    k, v, tabs = _ring_from_linear(case, ring)
    kw = case.oracle_kwargs()
    kw.update(k_cache=k, v_cache=v, block_tables=tabs)
    ref, ref_lse = oracle.paged_attention(**kw, sm_scale=1 / math.sqrt(d), window=window, ring_blocks=ring,
                                          nthreads=NTHREADS)
    for chunk in (0, 1, 4):
        out, lse = _decode(case, k, v, tabs, window, ring=ring, chunk=chunk)
        assert_close(out, ref, "ring decode chunk %d" % chunk)
        assert_lse_close(lse, ref_lse, "ring decode")
        lin, lin_lse = _decode(case, case.k_cache, case.v_cache, case.tables, window, chunk=chunk)
        assert torch.equal(out, lin) and torch.equal(lse, lin_lse), "ring and linear caches differ"
    assert pkv.pkv_device_errors() == 0


def test_ring_append_then_decode():
    """The last (up to) 144 tokens of each sequence appended (with RoPE) into a
    9-block ring, then decode with a 128-key window: equal to the oracle's
    append into a linear cache and its windowed attention."""
    rng = np.random.default_rng(52)
    hq, hkv, d, ring, window = 16, 2, 128, 9, 128
    lens = np.array([130, 1000, 4097, 144], np.int32)
    B = len(lens)
    n_new = np.minimum(lens, 144)  # the last (up to) 144 tokens: 9 ring blocks, each written once
    pos = np.concatenate([np.arange(L - n, L) for L, n in zip(lens, n_new)]).astype(np.int32)
    seq = np.repeat(np.arange(B), n_new).astype(np.int32)
    kn = rng.standard_normal((len(pos), hkv, d)).astype(np.float32)
    vn = rng.standard_normal((len(pos), hkv, d)).astype(np.float32)
    kb, vb = bf16_bits(kn), bf16_bits(vn)
    table = oracle.rope_table(1e6, d, int(lens.max()))
    # oracle: linear cache
    mb = int((lens.max() + BS - 1) // BS)
    lin_tabs = (np.arange(mb)[None, :] + mb * np.arange(B)[:, None]).astype(np.int32)
    lk = np.zeros((B * mb, hkv, BS, d), np.uint16)
    lv = np.zeros_like(lk)
    oracle.append_rope(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS, kv_dtype=oracle.KV_BF16,
                       k_cache=lk, v_cache=lv, block_tables=lin_tabs, token_to_seq=seq, positions=pos,
                       k_new=kb, v_new=vb, cos_sin=table)
    q = bf16_bits(rng.standard_normal((B, hq, d)).astype(np.float32))
    ref, ref_lse = oracle.paged_attention(q=q, k_cache=lk, v_cache=lv, block_tables=lin_tabs,
                                          qo_indptr=np.arange(B + 1), kv_lens=lens, num_q_heads=hq,
                                          num_kv_heads=hkv, sm_scale=1 / math.sqrt(d), window=window,
                                          nthreads=NTHREADS)
    # GPU: ring cache, one append call (144 tokens fill the 9 ring blocks exactly once)
    rtabs = (np.arange(ring)[None, :] + ring * np.arange(B)[:, None]).astype(np.int32)
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=B * ring,
                         max_blocks_per_seq=ring, ring_blocks=ring)
    rk = torch.zeros((B * ring, hkv, BS, d), dtype=torch.bfloat16, device=DEV)
    rv = torch.zeros_like(rk)
    pkv.pkv_append_rope(desc, rk, rv, _dev(rtabs), _dev(seq), _dev(pos), _dev_pool(kb), _dev_pool(vb),
                        cos_sin=_dev(table))
    out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, hq), device=DEV)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, int(lens.max()), window, 0), 256),
                     dtype=torch.uint8, device=DEV)
    pkv.pkv_decode_attention(desc, _dev_pool(q), rk, rv, _dev(rtabs), _dev(lens), int(lens.max()),
                             1 / math.sqrt(d), out, lse, ws, window=window)
    torch.cuda.synchronize()
    assert_close(out, ref, "ring append + decode")
    assert_lse_close(lse, ref_lse, "ring append + decode")
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("fp8,window", [(False, -1), (False, 128), (True, -1), (True, 128)])
def test_sinks_match_oracle(fp8, window):
    rng = np.random.default_rng(60 + 2 * fp8 + (window > 0))
    hq, hkv, d = (64, 8, 64) if fp8 else (16, 2, 128)
    case = PagedCase(rng, [1, 30, 128, 129, 500, 2048], hq, hkv, d, fp8=fp8)
    sinks = rng.uniform(-2.0, 6.0, hq).astype(np.float32)
    sinks[::5] = -np.inf
    ref, ref_lse = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=1 / math.sqrt(d), window=window,
                                          sinks=sinks, nthreads=NTHREADS)
    for chunk in (0, 1, 3):  # one chunk per sequence, and merged splits
        out, lse = _decode(case, case.k_cache, case.v_cache, case.tables, window, sinks=sinks, chunk=chunk)
        assert_close(out, ref, "sinks chunk %d" % chunk)
        assert_lse_close(lse, ref_lse, "sinks")
    out_s, lse_s = _decode(case, case.k_cache, case.v_cache, case.tables, window, sinks=sinks, static=True)
    assert_close(out_s, ref, "sinks, no-workspace entry")
    assert pkv.pkv_device_errors() == 0


def test_ring_with_sinks():
    rng = np.random.default_rng(70)
    case = PagedCase(rng, [5, 200, 2500], 32, 8, 128)
    k, v, tabs = _ring_from_linear(case, 9)
    kw = case.oracle_kwargs()
    kw.update(k_cache=k, v_cache=v, block_tables=tabs)
    sinks = rng.uniform(-1.0, 3.0, 32).astype(np.float32)
    ref, ref_lse = oracle.paged_attention(**kw, sm_scale=1 / math.sqrt(128), window=128, ring_blocks=9,
                                          sinks=sinks, nthreads=NTHREADS)
    out, lse = _decode(case, k, v, tabs, 128, ring=9, sinks=sinks)
    assert_close(out, ref, "ring + sinks")
    assert_lse_close(lse, ref_lse, "ring + sinks")
