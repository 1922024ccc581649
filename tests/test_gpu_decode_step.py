"""GPU parity of the fused decode step (llm-infer, "What It Does": KV writes
and fused RoPE inside the decode step): one launch appends every sequence's
new token (RoPE'd K, V; e4m3 quantised for FP8 pools), rotates q and attends.

Checked three ways on the same seeded bytes:
  * the cache after the step equals the oracle's append, byte for byte;
  * out / lse match the oracle's attention over that cache with the oracle's
    rotated q, within the attention tolerance;
  * out / lse / cache equal, bit for bit, the two-launch path (append with an
    in-place q rotation, then plain decode) -- the fusion changes no
    arithmetic."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._cases import BS, PagedCase, bf16_bits
from tests._gpu import (DEV, NTHREADS, assert_close, assert_lse_close, compact_pool, desc_for, on_device,
                        pool_np, u16)

pytestmark = pytest.mark.gpu

LENS = [1, 2, 15, 16, 17, 33, 64, 65, 129, 700, 2049, 4100]


def _pool(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if bits.dtype == np.uint16:
        return t.view(torch.int16).view(torch.bfloat16).to(DEV)
    return t.to(DEV)


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _setup(seed, lens, hq, hkv, d, fp8, rope):
    rng = np.random.default_rng(seed)
    case = PagedCase(rng, lens, hq, hkv, d, fp8=fp8)
    B = len(lens)
    k_new = bf16_bits(rng.standard_normal((B, hkv, d)).astype(np.float32))
    v_new = bf16_bits(rng.standard_normal((B, hkv, d)).astype(np.float32))
    table = oracle.rope_table(1e6, d, int(max(lens))) if rope else None
    return case, k_new, v_new, table


def _oracle_step(case, k_new, v_new, table, tables, k_cache, v_cache, window, ring=0, sinks=None):
    """Oracle: append at position len - 1 (rotating q), then attention."""
    B = len(case.lens)
    kc, vc = k_cache.copy(), v_cache.copy()
    q_rot = oracle.append_rope(num_q_heads=case.hq, num_kv_heads=case.hkv, head_dim=case.d,
                               block_size=BS, kv_dtype=1 if case.fp8 else 0, k_cache=kc, v_cache=vc,
                               block_tables=tables, token_to_seq=np.arange(B, dtype=np.int32),
                               positions=(case.lens - 1).astype(np.int32), k_new=k_new, v_new=v_new,
                               q=case.q, cos_sin=table, k_scale=case.k_scale, v_scale=case.v_scale,
                               ring_blocks=ring)
    ref, ref_lse = oracle.paged_attention(q=q_rot, k_cache=kc, v_cache=vc, block_tables=tables,
                                          qo_indptr=np.arange(B + 1), kv_lens=case.lens,
                                          num_q_heads=case.hq, num_kv_heads=case.hkv,
                                          sm_scale=1 / math.sqrt(case.d), window=window,
                                          kv_dtype=1 if case.fp8 else 0, k_scale=case.k_scale,
                                          v_scale=case.v_scale, ring_blocks=ring, sinks=sinks,
                                          nthreads=NTHREADS)
    return kc, vc, ref, ref_lse


def _gpu(case, k_new, v_new, table, tables, k_cache, v_cache, window, chunk, fused, ring=0,
         sinks=None, flags=0):
    B = len(case.lens)
    desc = pkv.make_desc(num_q_heads=case.hq, num_kv_heads=case.hkv, head_dim=case.d,
                         num_blocks=k_cache.shape[0], max_blocks_per_seq=tables.shape[1],
                         kv_dtype=1 if case.fp8 else 0, ring_blocks=ring, flags=flags)
    max_ctx = int(case.lens.max())
    kd, vd = _pool(k_cache), _pool(v_cache)
    q = _pool(case.q)
    out = torch.full((B, case.hq, case.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, case.hq), float("nan"), device=DEV)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, window, chunk), 256),
                     dtype=torch.uint8, device=DEV)
    lens = _dev(case.lens)
    tabs = _dev(tables)
    ks, vs, sk = _dev(case.k_scale), _dev(case.v_scale), _dev(sinks)
    cs = _dev(table)
    if fused:
        q_before = q.clone()
        pkv.pkv_decode_step(desc, q, _pool(k_new), _pool(v_new), kd, vd, tabs, lens, max_ctx,
                            1 / math.sqrt(case.d), out, lse, ws, cos_sin=cs, window=window,
                            chunk_blocks=chunk, k_scale=ks, v_scale=vs, sinks=sk)
        torch.cuda.synchronize()
        assert torch.equal(q, q_before), "the decode step must not modify q"
    else:
        pkv.pkv_append_rope(desc, kd, vd, tabs, _dev(np.arange(B, dtype=np.int32)),
                            _dev((case.lens - 1).astype(np.int32)), _pool(k_new), _pool(v_new), q=q,
                            cos_sin=cs, k_scale=ks, v_scale=vs)
        pkv.pkv_decode_attention(desc, q, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(case.d), out, lse,
                                 ws, window=window, chunk_blocks=chunk, k_scale=ks, v_scale=vs,
                                 sinks=sk)
        torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    assert int(ws[:4 * B * case.hkv].view(torch.int32).abs().sum().item()) == 0, "tickets not reset"
    return out, lse, kd, vd


@pytest.mark.parametrize("hq,hkv,d,fp8", [(16, 2, 128, False), (32, 8, 128, False), (8, 2, 64, False),
                                          (64, 8, 64, True), (16, 2, 128, True), (16, 4, 64, False),
                                          (32, 8, 128, True)])
@pytest.mark.parametrize("rope", [True, False])
def test_decode_step_matches_oracle_and_two_launch_path(hq, hkv, d, fp8, rope):
    case, k_new, v_new, table = _setup(80 + d + hq + fp8, LENS, hq, hkv, d, fp8, rope)
    kc, vc, ref, ref_lse = _oracle_step(case, k_new, v_new, table, case.tables, case.k_cache,
                                        case.v_cache, -1)
    for chunk in (0, 1, 3):
        out, lse, kd, vd = _gpu(case, k_new, v_new, table, case.tables, case.k_cache, case.v_cache,
                                -1, chunk, fused=True)
        assert np.array_equal(pool_np(kd), kc), "K cache after the step differs from the oracle's append"
        assert np.array_equal(pool_np(vd), vc), "V cache after the step differs from the oracle's append"
        assert_close(out, ref, "decode step %d/%d/%d fp8=%d chunk %d" % (hq, hkv, d, fp8, chunk))
        assert_lse_close(lse, ref_lse, "decode step lse")
        out2, lse2, kd2, vd2 = _gpu(case, k_new, v_new, table, case.tables, case.k_cache, case.v_cache,
                                    -1, chunk, fused=False)
        assert torch.equal(out, out2) and torch.equal(lse, lse2), "fused and two-launch outputs differ"
        assert torch.equal(kd, kd2) and torch.equal(vd, vd2), "fused and two-launch caches differ"


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("flags", [0, pkv.DESC_PREFETCH_KV])
def test_decode_step_window_sinks_ring(fp8, flags):
    """Sliding window 128 over a 9-block ring, with sink logits: the step
    writes into ring entry ((len - 1) / 16) mod 9.  With PKV_DESC_PREFETCH_KV
    the ring entries and the first blocks are read before the wait."""
    hq, hkv, d = (64, 8, 64) if fp8 else (32, 8, 128)
    case, k_new, v_new, table = _setup(90 + fp8, [1, 16, 17, 128, 129, 145, 1000, 3001], hq, hkv, d,
                                       fp8, True)
    ring = 9
    B = len(case.lens)
    rk = np.zeros((B * ring,) + case.k_cache.shape[1:], case.k_cache.dtype)
    rv = np.zeros_like(rk)
    rtabs = (np.arange(ring)[None, :] + ring * np.arange(B)[:, None]).astype(np.int32)
    for s in range(B):
        for b in range((int(case.lens[s]) + BS - 1) // BS):
            rk[rtabs[s, b % ring]] = case.k_cache[case.tables[s, b]]
            rv[rtabs[s, b % ring]] = case.v_cache[case.tables[s, b]]
    rng = np.random.default_rng(7)
    sinks = rng.uniform(-1.0, 4.0, hq).astype(np.float32)
    kc, vc, ref, ref_lse = _oracle_step(case, k_new, v_new, table, rtabs, rk, rv, 128, ring=ring,
                                        sinks=sinks)
    for chunk in (0, 2):
        out, lse, kd, vd = _gpu(case, k_new, v_new, table, rtabs, rk, rv, 128, chunk, fused=True,
                                ring=ring, sinks=sinks, flags=flags)
        assert np.array_equal(pool_np(kd), kc) and np.array_equal(pool_np(vd), vc)
        assert_close(out, ref, "ring step chunk %d" % chunk)
        assert_lse_close(lse, ref_lse, "ring step lse")
        out2, lse2, _, _ = _gpu(case, k_new, v_new, table, rtabs, rk, rv, 128, chunk, fused=False,
                                ring=ring, sinks=sinks)
        assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_decode_step_in_a_graph_repeats():
    """Replaying a captured step rewrites the same slots with the same bytes:
    the cache and the output are those of one step, however many replays."""
    case, k_new, v_new, table = _setup(95, [5, 300, 1024, 2500], 16, 2, 128, False, True)
    kc, vc, ref, ref_lse = _oracle_step(case, k_new, v_new, table, case.tables, case.k_cache,
                                        case.v_cache, -1)
    B = len(case.lens)
    desc = pkv.make_desc(num_q_heads=16, num_kv_heads=2, head_dim=128, num_blocks=case.k_cache.shape[0],
                         max_blocks_per_seq=case.tables.shape[1])
    max_ctx = int(case.lens.max())
    kd, vd, q = _pool(case.k_cache), _pool(case.v_cache), _pool(case.q)
    kn, vn, cs = _pool(k_new), _pool(v_new), _dev(table)
    tabs, lens = _dev(case.tables), _dev(case.lens)
    out = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, 16), device=DEV)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, 2), 256), dtype=torch.uint8,
                     device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.pkv_decode_step(desc, q, kn, vn, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(128), out, lse, ws,
                            cos_sin=cs, chunk_blocks=2, stream=s)  # warm-up (attribute set)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.pkv_decode_step(desc, q, kn, vn, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(128), out, lse, ws,
                            cos_sin=cs, chunk_blocks=2, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(pool_np(kd), kc) and np.array_equal(pool_np(vd), vc)
    assert_close(out, ref, "graph-replayed step")
    assert_lse_close(lse, ref_lse, "graph-replayed step")
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("hq,hkv,d,fp8", [(16, 2, 128, False), (64, 8, 64, True), (32, 8, 128, False)])
def test_prefetch_kv_steps_back_to_back_match_oracle(hq, hkv, d, fp8):
    """PKV_DESC_PREFETCH_KV: a step reads its lengths and block ids and
    starts its first K/V loads before the previous kernel on the stream has
    finished, and waits for it before touching q, k_new, v_new or writing.
    Two batches over separate pools alternate on one stream (each step's
    predecessor writes only the other batch's pools, as the promise asks),
    launched directly and replayed from a graph: every step's cache and
    output equal the oracle's, for planned, 1-block and 3-block chunks (the
    new token's block inside and outside each warp's first ring loads)."""
    cases = [_setup(210 + i + d + fp8, LENS, hq, hkv, d, fp8, True) for i in range(2)]
    refs = [_oracle_step(c, kn, vn, t, c.tables, c.k_cache, c.v_cache, -1) for (c, kn, vn, t) in cases]
    B = len(LENS)
    for chunk in (0, 1, 3):
        runs = []
        for (case, k_new, v_new, table) in cases:
            desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 num_blocks=case.k_cache.shape[0], max_blocks_per_seq=case.tables.shape[1],
                                 kv_dtype=1 if fp8 else 0, flags=pkv.DESC_PREFETCH_KV)
            max_ctx = int(case.lens.max())
            runs.append(dict(
                desc=desc, max_ctx=max_ctx, kd=_pool(case.k_cache), vd=_pool(case.v_cache), q=_pool(case.q),
                kn=_pool(k_new), vn=_pool(v_new), cs=_dev(table), tabs=_dev(case.tables),
                lens=_dev(case.lens), ks=_dev(case.k_scale), vs=_dev(case.v_scale),
                out=torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV),
                lse=torch.full((B, hq), float("nan"), device=DEV),
                ws=torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, chunk), 256),
                               dtype=torch.uint8, device=DEV)))
        s = torch.cuda.Stream()

        def step(r):
            pkv.pkv_decode_step(r["desc"], r["q"], r["kn"], r["vn"], r["kd"], r["vd"], r["tabs"], r["lens"],
                                r["max_ctx"], 1 / math.sqrt(d), r["out"], r["lse"], r["ws"], cos_sin=r["cs"],
                                chunk_blocks=chunk, k_scale=r["ks"], v_scale=r["vs"], stream=s)

        with torch.cuda.stream(s):
            for _ in range(3):
                for r in runs:
                    step(r)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(2):
                for r in runs:
                    step(r)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert pkv.pkv_device_errors() == 0
        for r, (kc, vc, ref, ref_lse) in zip(runs, refs):
            assert np.array_equal(pool_np(r["kd"]), kc) and np.array_equal(pool_np(r["vd"]), vc), \
                "cache after prefetching steps differs from the oracle's append"
            assert_close(r["out"], ref, "prefetching step %d/%d/%d fp8=%d chunk %d" % (hq, hkv, d, fp8, chunk))
            assert_lse_close(r["lse"], ref_lse, "prefetching step lse")
            assert int(r["ws"][:4 * B * hkv].view(torch.int32).abs().sum().item()) == 0, "tickets not reset"


def test_prefetch_kv_alternating_batches_growing_steps():
    """Two batches alternate on one stream for four steps each, with
    PKV_DESC_PREFETCH_KV and growing lengths: step t of a batch appends at
    position len + t - 1 and reads the row its own step t - 1 appended, two
    launches earlier (the other batch's step in between, as the promise
    allows).  Every step's output equals the oracle's step-by-step append and
    attention."""
    hq, hkv, d = 16, 2, 128
    steps = 4
    runs = []
    for i in range(2):
        rng = np.random.default_rng(240 + i)
        lens = np.array([4, 17, 33, 130, 700, 2050], dtype=np.int32)
        case = PagedCase(rng, lens, hq, hkv, d)
        B = len(lens)
        k_new = [bf16_bits(rng.standard_normal((B, hkv, d)).astype(np.float32)) for _ in range(steps)]
        v_new = [bf16_bits(rng.standard_normal((B, hkv, d)).astype(np.float32)) for _ in range(steps)]
        qs = [bf16_bits(rng.standard_normal((B, hq, d)).astype(np.float32)) for _ in range(steps)]
        table = oracle.rope_table(1e6, d, int(lens.max()))
        # the oracle, step by step on one host copy of the cache
        kc, vc = case.k_cache.copy(), case.v_cache.copy()
        refs = []
        for t in range(steps):
            lt = (lens - steps + 1 + t).astype(np.int32)
            q_rot = oracle.append_rope(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS, kv_dtype=0,
                                       k_cache=kc, v_cache=vc, block_tables=case.tables,
                                       token_to_seq=np.arange(B, dtype=np.int32), positions=lt - 1,
                                       k_new=k_new[t], v_new=v_new[t], q=qs[t], cos_sin=table)
            refs.append(oracle.paged_attention(q=q_rot, k_cache=kc, v_cache=vc, block_tables=case.tables,
                                               qo_indptr=np.arange(B + 1), kv_lens=lt, num_q_heads=hq,
                                               num_kv_heads=hkv, sm_scale=1 / math.sqrt(d), nthreads=NTHREADS))
        desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=case.k_cache.shape[0],
                             max_blocks_per_seq=case.tables.shape[1], flags=pkv.DESC_PREFETCH_KV)
        max_ctx = int(lens.max())
        runs.append(dict(
            desc=desc, max_ctx=max_ctx, refs=refs, kd=_pool(case.k_cache), vd=_pool(case.v_cache),
            q=[_pool(x) for x in qs], kn=[_pool(x) for x in k_new], vn=[_pool(x) for x in v_new],
            lens=[_dev((lens - steps + 1 + t).astype(np.int32)) for t in range(steps)], tabs=_dev(case.tables),
            cs=_dev(table), out=[torch.empty((B, hq, d), dtype=torch.bfloat16, device=DEV) for _ in range(steps)],
            lse=[torch.empty((B, hq), device=DEV) for _ in range(steps)],
            ws=torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, 2), 256), dtype=torch.uint8,
                           device=DEV)))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for t in range(steps):
            for r in runs:
                pkv.pkv_decode_step(r["desc"], r["q"][t], r["kn"][t], r["vn"][t], r["kd"], r["vd"], r["tabs"],
                                    r["lens"][t], r["max_ctx"], 1 / math.sqrt(d), r["out"][t], r["lse"][t], r["ws"],
                                    cos_sin=r["cs"], chunk_blocks=2, stream=s)
    s.synchronize()
    assert pkv.pkv_device_errors() == 0
    for i, r in enumerate(runs):
        for t in range(steps):
            ref, ref_lse = r["refs"][t]
            assert_close(r["out"][t], ref, "alternating batch %d, step %d" % (i, t))
            assert_lse_close(r["lse"][t], ref_lse, "alternating batch %d, step %d" % (i, t))


def test_independent_decode_step_after_prefill_matches_oracle():
    """PKV_DESC_INDEPENDENT, one layer's mixed step: a ragged causal prefill
    (its own pools) and then the decode step of other sequences, which does
    not wait for the prefill and waits only at its end.  Alternating on one
    stream, directly and replayed from a graph, both outputs and the decode's
    cache equal the oracle's."""
    from tests.test_gpu_prefill import _oracle_prefill
    spec = wl.dataclasses.replace(wl.LLAMA3_8B_PREFILL, num_chunks=4, chunk_len=96, prefix_hi=700, seed=5)
    pb = wl.make_prefill_batch(spec, "cpu")
    p_ref, p_ref_lse = _oracle_prefill(spec, pb)
    pdesc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                          head_dim=spec.head_dim, num_blocks=pb.k_cache.shape[0],
                          max_blocks_per_seq=pb.tables_host.shape[1])
    pq, pk, pv = pb.q.to(DEV), pb.k_cache.to(DEV), pb.v_cache.to(DEV)
    pqo, pkvl, ptab = (torch.from_numpy(x).to(DEV) for x in (pb.qo_indptr_host, pb.kv_lens_host, pb.tables_host))
    p_out = torch.full((pb.total_q, spec.num_q_heads, spec.head_dim), float("nan"), dtype=torch.bfloat16,
                       device=DEV)
    p_lse = torch.full((pb.total_q, spec.num_q_heads), float("nan"), device=DEV)

    hq, hkv, d = 32, 8, 128
    case, k_new, v_new, table = _setup(230, LENS, hq, hkv, d, False, True)
    kc, vc, ref, ref_lse = _oracle_step(case, k_new, v_new, table, case.tables, case.k_cache, case.v_cache, -1)
    B = len(LENS)
    for chunk in (0, 3):
        desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=case.k_cache.shape[0],
                             max_blocks_per_seq=case.tables.shape[1],
                             flags=pkv.DESC_INDEPENDENT | pkv.DESC_PREFETCH_KV)
        max_ctx = int(case.lens.max())
        kd, vd, q = _pool(case.k_cache), _pool(case.v_cache), _pool(case.q)
        kn, vn, cs = _pool(k_new), _pool(v_new), _dev(table)
        tabs, lens = _dev(case.tables), _dev(case.lens)
        out = torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, hq), float("nan"), device=DEV)
        ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, chunk), 256),
                         dtype=torch.uint8, device=DEV)
        s = torch.cuda.Stream()

        def mixed():
            pkv.pkv_prefill_attention_ragged(pdesc, pq, pqo, pk, pv, ptab, pkvl, spec.sm_scale, p_out, p_lse,
                                             qo_indptr_host=pb.qo_indptr_host, kv_lens_host=pb.kv_lens_host,
                                             stream=s)
            pkv.pkv_decode_step(desc, q, kn, vn, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(d), out, lse, ws,
                                cos_sin=cs, chunk_blocks=chunk, stream=s)

        with torch.cuda.stream(s):
            for _ in range(3):
                mixed()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(2):
                mixed()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert pkv.pkv_device_errors() == 0
        assert np.array_equal(pool_np(kd), kc) and np.array_equal(pool_np(vd), vc)
        assert_close(out, ref, "independent decode step chunk %d" % chunk)
        assert_lse_close(lse, ref_lse, "independent decode step lse")
        assert_close(p_out, p_ref, "prefill before an independent decode step")
        assert_lse_close(p_lse, p_ref_lse, "prefill lse")
        assert int(ws[:4 * B * hkv].view(torch.int32).abs().sum().item()) == 0, "tickets not reset"


def test_bound_decode_step_equals_the_unbound_call():
    """bind_decode_step marshals the arguments once; refilling the bound q
    and calling again gives the bits of a fresh unbound call."""
    case, k_new, v_new, table = _setup(97, [40, 300, 1024, 2500], 16, 2, 128, False, True)
    B = len(case.lens)
    desc = pkv.make_desc(num_q_heads=16, num_kv_heads=2, head_dim=128, num_blocks=case.k_cache.shape[0],
                         max_blocks_per_seq=case.tables.shape[1])
    max_ctx = int(case.lens.max())
    kn, vn, cs = _pool(k_new), _pool(v_new), _dev(table)
    tabs, lens = _dev(case.tables), _dev(case.lens)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, 0), 256), dtype=torch.uint8,
                     device=DEV)
    rng = np.random.default_rng(98)
    for trial in range(2):
        q_new = _pool(bf16_bits(rng.standard_normal((B, 16, 128)).astype(np.float32)))
        # unbound on fresh caches
        kd, vd = _pool(case.k_cache), _pool(case.v_cache)
        out_u = torch.empty((B, 16, 128), dtype=torch.bfloat16, device=DEV)
        pkv.pkv_decode_step(desc, q_new, kn, vn, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(128), out_u,
                            None, ws, cos_sin=cs)
        # bound on fresh caches: q written into the bound buffer first
        kd2, vd2 = _pool(case.k_cache), _pool(case.v_cache)
        if trial == 0:
            q_buf = torch.empty_like(q_new)
            out_b = torch.empty_like(out_u)
            call = pkv.bind_decode_step(desc, q_buf, kn, vn, kd2, vd2, tabs, lens, max_ctx,
                                        1 / math.sqrt(128), out_b, None, ws, cos_sin=cs)
        else:
            # the bound caches are the first trial's: refill them in place
            call._keep[4].copy_(kd2)
            call._keep[5].copy_(vd2)
        q_buf.copy_(q_new)
        call()
        torch.cuda.synchronize()
        assert torch.equal(out_b, out_u)
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("cfg,window", [(2, -1), (3, -1), (5, -1), (5, wl.FP8_WINDOW)])
def test_full_size_decode_step_on_sampled_sequences(cfg, window):
    """The full-size batches in the benchmark's launch configuration (one
    planned decode-step launch, inputs generated on the GPU).  A sample of
    sequences -- shortest, longest and random ones -- is checked against the
    oracle's own append and attention on a host copy of just their blocks,
    and their appended cache rows byte for byte."""
    spec = wl.CONFIGS[cfg]
    b = wl.make_decode_batch(spec, DEV)
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    max_ctx = b.max_context_len
    rng = np.random.default_rng(100 + cfg)
    seqs = sorted(set([int(np.argmin(b.lens_host)), int(np.argmax(b.lens_host))] +
                      rng.choice(spec.batch, size=4, replace=False).tolist()))
    k0, v0, tabs = compact_pool(d["k_cache"], d["v_cache"], b.tables_host, seqs)  # before the step
    table = pkv.pkv_rope_cos_sin_table(spec.rope_theta, spec.head_dim, max_ctx)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, spec.batch, max_ctx, window, 0), 256),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=DEV)
    pkv.pkv_decode_step(desc, d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["block_tables"],
                        d["context_lens"], max_ctx, spec.sm_scale, out, lse, ws,
                        cos_sin=torch.from_numpy(table).to(DEV), window=window, k_scale=d["k_scale"],
                        v_scale=d["v_scale"])
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    fp8 = spec.kv_dtype == "fp8_e4m3"
    ks = None if d["k_scale"] is None else d["k_scale"].cpu().numpy()
    vs = None if d["v_scale"] is None else d["v_scale"].cpu().numpy()
    lens = b.lens_host[seqs]
    q_rot = oracle.append_rope(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                               head_dim=spec.head_dim, block_size=BS, kv_dtype=1 if fp8 else 0,
                               k_cache=k0, v_cache=v0, block_tables=tabs,
                               token_to_seq=np.arange(len(seqs), dtype=np.int32),
                               positions=(lens - 1).astype(np.int32), k_new=u16(d["k_new"])[seqs],
                               v_new=u16(d["v_new"])[seqs], q=u16(d["q"])[seqs],
                               cos_sin=oracle.rope_table(spec.rope_theta, spec.head_dim, max_ctx),
                               k_scale=ks, v_scale=vs)
    k1, v1, _ = compact_pool(d["k_cache"], d["v_cache"], b.tables_host, seqs)  # after the step
    assert np.array_equal(k1, k0) and np.array_equal(v1, v0), "appended rows differ from the oracle's"
    ref, ref_lse = oracle.paged_attention(q=q_rot, k_cache=k0, v_cache=v0, block_tables=tabs,
                                          qo_indptr=np.arange(len(seqs) + 1), kv_lens=lens,
                                          num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                          sm_scale=spec.sm_scale, window=window, kv_dtype=1 if fp8 else 0,
                                          k_scale=ks, v_scale=vs, nthreads=NTHREADS)
    assert_close(out[seqs], ref, "%s decode step, sampled" % spec.name)
    assert_lse_close(lse[seqs], ref_lse, "%s decode step" % spec.name)


@pytest.mark.parametrize("fp8", [False, True])
def test_pinned_host_inputs_and_outputs_give_the_same_bytes(fp8):
    """The per-step arrays (q, k_new, v_new, tables, lengths, out, lse) in
    pinned host memory, read and written by the kernel over the host link:
    the cache, out and lse equal the all-device call bit for bit."""
    hq, hkv, d = (16, 2, 128) if not fp8 else (64, 8, 64)
    case, k_new, v_new, table = _setup(321 + fp8, LENS, hq, hkv, d, fp8, True)
    B = len(case.lens)
    max_ctx = int(case.lens.max())
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=case.k_cache.shape[0],
                         max_blocks_per_seq=case.tables.shape[1], kv_dtype=1 if fp8 else 0)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, 0), 256), dtype=torch.uint8,
                     device=DEV)
    cs = _dev(table)
    ks, vs = _dev(case.k_scale), _dev(case.v_scale)
    results = []
    for host in (False, True):
        put = (lambda t: t.cpu().contiguous().pin_memory()) if host else (lambda t: t)
        q = put(_pool(case.q))
        kn, vn = put(_pool(k_new)), put(_pool(v_new))
        tabs, lens = put(_dev(case.tables)), put(_dev(case.lens))
        kd, vd = _pool(case.k_cache), _pool(case.v_cache)
        out = put(torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV))
        lse = put(torch.full((B, hq), float("nan"), device=DEV))
        pkv.pkv_decode_step(desc, q, kn, vn, kd, vd, tabs, lens, max_ctx, 1 / math.sqrt(d), out, lse, ws,
                            cos_sin=cs, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        assert pkv.pkv_device_errors() == 0
        results.append((out.cpu(), lse.cpu(), kd.cpu(), vd.cpu()))
    for a, b in zip(*results):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
