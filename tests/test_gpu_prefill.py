"""GPU parity of ragged causal chunked prefill over cached prefixes, plus the
invariants the pages state: chunked == one-shot, prefix-cached (shared
blocks) == private copies, decode == one-token prefill."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import (DEV, NTHREADS, assert_close, assert_lse_close, compact_pool, gpu_decode,
                        pool_np, u16)

pytestmark = pytest.mark.gpu


def _desc(spec, k_cache, tables):
    return pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=k_cache.shape[0],
                         max_blocks_per_seq=tables.shape[1])


def _gpu_prefill(spec, pb, q=None, qo=None, kvl=None, tables=None, causal=True, window=-1,
                 k_cache=None, v_cache=None):
    q = pb.q if q is None else q
    qo = pb.qo_indptr_host if qo is None else qo
    kvl = pb.kv_lens_host if kvl is None else kvl
    tables = pb.tables_host if tables is None else tables
    kc = (pb.k_cache if k_cache is None else k_cache).to(DEV)
    vc = (pb.v_cache if v_cache is None else v_cache).to(DEV)
    desc = _desc(spec, kc, tables)
    out = torch.full((q.shape[0], spec.num_q_heads, spec.head_dim), float("nan"),
                     dtype=torch.bfloat16, device=DEV)
    lse = torch.full((q.shape[0], spec.num_q_heads), float("nan"), device=DEV)
    pkv.pkv_prefill_attention_ragged(desc, q.to(DEV), torch.from_numpy(qo).to(DEV), kc, vc,
                                     torch.from_numpy(tables).to(DEV),
                                     torch.from_numpy(kvl).to(DEV), spec.sm_scale, out, lse,
                                     qo_indptr_host=qo, kv_lens_host=kvl, causal=causal,
                                     window=window)
    torch.cuda.synchronize()
    return out, lse


def _oracle_prefill(spec, pb, q=None, qo=None, kvl=None, tables=None, causal=True, window=-1,
                    k_np=None, v_np=None):
    return oracle.paged_attention(
        q=u16(pb.q if q is None else q),
        k_cache=pool_np(pb.k_cache) if k_np is None else k_np,
        v_cache=pool_np(pb.v_cache) if v_np is None else v_np,
        block_tables=pb.tables_host if tables is None else tables,
        qo_indptr=pb.qo_indptr_host if qo is None else qo,
        kv_lens=pb.kv_lens_host if kvl is None else kvl, num_q_heads=spec.num_q_heads,
        num_kv_heads=spec.num_kv_heads, sm_scale=spec.sm_scale, causal=causal, window=window,
        nthreads=NTHREADS)


def _small(num_chunks=4, chunk=96, hq=32, hkv=8, d=128, prefix_hi=700, seed=3):
    return wl.PrefillSpec("prefill small", num_chunks=num_chunks, chunk_len=chunk, prefix_lo=0,
                          prefix_hi=prefix_hi, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                          seed=seed)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (16, 2, 128), (8, 2, 64), (4, 4, 64),
                                      (12, 4, 128)])
def test_ragged_causal_prefill_matches_oracle(hq, hkv, d):
    spec = _small(hq=hq, hkv=hkv, d=d)
    q_lens = [96, 1, 37, 130]
    prefixes = [0, 0, 515, 515]
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=q_lens, prefixes=prefixes)
    out, lse = _gpu_prefill(spec, pb)
    ref, ref_lse = _oracle_prefill(spec, pb)
    assert_close(out, ref, "prefill %d/%d/%d" % (hq, hkv, d))
    assert_lse_close(lse, ref_lse, "prefill")
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("causal,window", [(False, -1), (True, 128), (True, 1), (True, 40)])
def test_prefill_masks(causal, window):
    spec = _small()
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[70, 200, 5, 64], prefixes=[300, 300, 33, 33])
    out, lse = _gpu_prefill(spec, pb, causal=causal, window=window)
    ref, ref_lse = _oracle_prefill(spec, pb, causal=causal, window=window)
    assert_close(out, ref, "prefill causal=%s window=%d" % (causal, window))
    assert_lse_close(lse, ref_lse, "prefill masks")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (16, 2, 128), (64, 8, 64)])
def test_short_multi_token_queries(hq, hkv, d):
    """Speculative-verify shapes (infer-lab, "Technique" table: speculative
    decoding): 2-8 new tokens per sequence after a long cached context, run
    through the ragged prefill kernel and checked against the oracle."""
    spec = _small(num_chunks=12, hq=hq, hkv=hkv, d=d, prefix_hi=3000, seed=11)
    rng = np.random.default_rng(11)
    q_lens = [int(v) for v in rng.integers(2, 9, 12)]
    prefixes = [int(v) for v in np.repeat(rng.integers(100, 3001, 6), 2)]
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=q_lens, prefixes=prefixes)
    out, lse = _gpu_prefill(spec, pb)
    ref, ref_lse = _oracle_prefill(spec, pb)
    assert_close(out, ref, "verify q_len 2-8, %d/%d/%d" % (hq, hkv, d))
    assert_lse_close(lse, ref_lse, "verify")
    assert pkv.pkv_device_errors() == 0


def test_chunked_prefill_equals_one_shot():
    """infer-lab's invariant: chunked prefill == one-shot prefill.  The oracle
    holds it bit for bit; the kernel within the attention tolerance."""
    spec = _small(num_chunks=2)
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[300, 300], prefixes=[0, 0])
    one, _ = _gpu_prefill(spec, pb)
    pieces = []
    for a, b in ((0, 64), (64, 65), (65, 200), (200, 300)):
        qo = np.array([0, b - a], np.int32)
        kvl = np.array([b], np.int32)
        o, _ = _gpu_prefill(spec, pb, q=pb.q[a:b], qo=qo, kvl=kvl, tables=pb.tables_host[:1])
        pieces.append(o)
    chunked = torch.cat(pieces)
    err = (chunked.float() - one[:300].float()).abs()
    assert err.max().item() <= 1e-2 and err.mean().item() <= 1e-3


def test_shared_prefix_blocks_equal_private_copies():
    spec = _small(num_chunks=2)
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[50, 50], prefixes=[400, 400])
    # sequence 1 shares sequence 0's 25 full prefix blocks; give it private copies
    shared = 400 // 16
    nb = pb.k_cache.shape[0]
    kc = torch.cat([pb.k_cache, torch.zeros_like(pb.k_cache[:shared])])
    vc = torch.cat([pb.v_cache, torch.zeros_like(pb.v_cache[:shared])])
    tabs = pb.tables_host.copy()
    free = list(range(nb, nb + shared))  # fresh blocks appended to the pool
    assert np.array_equal(tabs[0, :shared], tabs[1, :shared])
    for j in range(shared):
        kc[free[j]] = kc[tabs[1, j]]
        vc[free[j]] = vc[tabs[1, j]]
        tabs[1, j] = free[j]
    shared_out, _ = _gpu_prefill(spec, pb)
    private_out, _ = _gpu_prefill(spec, pb, tables=tabs, k_cache=kc, v_cache=vc)
    assert torch.equal(shared_out, private_out)


def test_decode_equals_one_token_prefill():
    spec = wl.scaled(wl.QWEN3_4B, batch=12, ctx_hi=700)
    b = wl.make_decode_batch(spec, "cpu")
    desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=b.k_cache.shape[0],
                         max_blocks_per_seq=b.tables_host.shape[1])
    d = dict(q=b.q.to(DEV), k_cache=b.k_cache.to(DEV), v_cache=b.v_cache.to(DEV), k_scale=None,
             v_scale=None, block_tables=b.block_tables.to(DEV), context_lens=b.context_lens.to(DEV))
    dec, dec_lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
    pspec = wl.PrefillSpec("one-token", num_chunks=12, chunk_len=1, prefix_lo=0, prefix_hi=0,
                           num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                           head_dim=spec.head_dim, seed=0)
    qo = np.arange(13, dtype=np.int32)
    out = torch.empty_like(d["q"])
    lse = torch.empty(dec_lse.shape, device=DEV)
    pkv.pkv_prefill_attention_ragged(desc, d["q"], torch.from_numpy(qo).to(DEV), d["k_cache"],
                                     d["v_cache"], d["block_tables"], d["context_lens"],
                                     spec.sm_scale, out, lse, qo_indptr_host=qo,
                                     kv_lens_host=b.lens_host)
    torch.cuda.synchronize()
    err = (out.float() - dec.float()).abs()
    assert err.max().item() <= 1e-2 and err.mean().item() <= 1e-3
    assert (lse - dec_lse).abs().max().item() <= 2e-3
    del pspec


def test_mixed_step_workload_full_size():
    """The Llama-3-8B-shaped mixed step at full size: 8 chunks of 512 tokens
    over shared prefixes of 0-8192, checked token by token against the oracle
    on two of the four pairs."""
    spec = wl.LLAMA3_8B_PREFILL
    pb = wl.make_prefill_batch(spec, DEV)
    out, lse = _gpu_prefill(spec, pb)
    seqs = [int(np.argmax(pb.prefix_host)), int(np.argmin(pb.prefix_host))]
    seqs = sorted(set(seqs))
    k, v, tabs = compact_pool(pb.k_cache, pb.v_cache, pb.tables_host, seqs)
    qo = pb.qo_indptr_host
    rows = np.concatenate([np.arange(qo[s], qo[s + 1]) for s in seqs])
    sub_qo = np.concatenate([[0], np.cumsum([qo[s + 1] - qo[s] for s in seqs])]).astype(np.int32)
    ref, ref_lse = oracle.paged_attention(q=u16(pb.q)[rows], k_cache=k, v_cache=v,
                                          block_tables=tabs, qo_indptr=sub_qo,
                                          kv_lens=pb.kv_lens_host[seqs],
                                          num_q_heads=spec.num_q_heads,
                                          num_kv_heads=spec.num_kv_heads, sm_scale=spec.sm_scale,
                                          nthreads=NTHREADS)
    assert_close(out[torch.from_numpy(rows).to(DEV)], ref, "mixed-step prefill")
    assert_lse_close(lse[torch.from_numpy(rows).to(DEV)], ref_lse, "mixed-step prefill")
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("hq,hkv,d,window,short", [(32, 8, 128, -1, False), (64, 8, 64, -1, False),
                                                   (16, 2, 128, 128, False), (64, 8, 64, 128, False),
                                                   (32, 8, 128, -1, True), (64, 8, 64, 128, True)])
def test_fp8_prefill_matches_oracle(hq, hkv, d, window, short):
    """Ragged causal prefill over e4m3 pools with per-head scales (InferX, "The
    kernels underneath": FP8 KV cache): against the oracle on the same codes.
    short: at most 64 query rows per sequence, so the short-query kernel
    converts the codes into its MMA fragments; otherwise the tcgen05 kernel
    converts the tiles in shared memory.  Neither takes a workspace."""
    from tests._cases import PagedCase
    rng = np.random.default_rng(80 + d + hq + (window > 0) + 7 * short)
    q_lens = [min(8, 64 // (hq // hkv)), 1, 3, 1, 1] if short else [64, 200, 77, 1, 1]
    case = PagedCase(rng, [300, 1000, 77, 520, 1], hq, hkv, d, q_lens=q_lens, fp8=True)
    sm = 1.0 / np.sqrt(d)
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=case.num_blocks,
                         max_blocks_per_seq=case.mbps, kv_dtype=pkv.KV_FP8_E4M3)
    T = int(case.qo[-1])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    q = t(case.q).view(torch.int16).view(torch.bfloat16) if case.q.dtype == np.uint16 else t(case.q)
    out = torch.full((T, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, hq), float("nan"), device=DEV)
    assert pkv.pkv_prefill_workspace_size(desc, len(case.lens), T) == 0
    ws = None
    for _ in range(2):  # two calls in a row
        pkv.pkv_prefill_attention_ragged(desc, q, t(case.qo), t(case.k_cache), t(case.v_cache), t(case.tables),
                                         t(case.lens), sm, out, lse, qo_indptr_host=case.qo,
                                         kv_lens_host=case.lens, window=window, workspace=ws,
                                         k_scale=t(case.k_scale), v_scale=t(case.v_scale))
        torch.cuda.synchronize()
        ref, ref_lse = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=sm, causal=True, window=window,
                                              nthreads=NTHREADS)
        assert_close(out, ref, "fp8 prefill %d/%d/%d" % (hq, hkv, d))
        assert_lse_close(lse, ref_lse, "fp8 prefill")
    assert pkv.pkv_device_errors() == 0


def test_fp8_mixed_step_workload_full_size():
    """The Llama-3-8B-shaped prefill part over e4m3 pools (per-head scales: each
    head's largest |value| / 448) through the tcgen05 kernel, which converts
    the tiles in shared memory and takes no workspace: token by token against
    the oracle on the same codes, for the longest and the shortest prefix."""
    spec = wl.LLAMA3_8B_PREFILL
    pb = wl.make_prefill_batch(spec, DEV)
    ks = (pb.k_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
    vs = (pb.v_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
    k8 = (pb.k_cache.float() / ks.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (pb.v_cache.float() / vs.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=k8.shape[0],
                         max_blocks_per_seq=pb.tables_host.shape[1], kv_dtype=pkv.KV_FP8_E4M3)
    out = torch.full_like(pb.q, float("nan"))
    lse = torch.full(pb.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pkv.pkv_device_errors(reset=True)
    pkv.pkv_prefill_attention_ragged(desc, pb.q, pb.qo_indptr, k8, v8, pb.block_tables, pb.kv_lens,
                                     spec.sm_scale, out, lse, qo_indptr_host=pb.qo_indptr_host,
                                     kv_lens_host=pb.kv_lens_host, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    seqs = sorted({int(np.argmax(pb.prefix_host)), int(np.argmin(pb.prefix_host))})
    k, v, tabs = compact_pool(k8, v8, pb.tables_host, seqs)
    qo = pb.qo_indptr_host
    rows = np.concatenate([np.arange(qo[s], qo[s + 1]) for s in seqs])
    sub_qo = np.concatenate([[0], np.cumsum([qo[s + 1] - qo[s] for s in seqs])]).astype(np.int32)
    ref, ref_lse = oracle.paged_attention(q=u16(pb.q)[rows], k_cache=k, v_cache=v, block_tables=tabs,
                                          qo_indptr=sub_qo, kv_lens=pb.kv_lens_host[seqs],
                                          num_q_heads=spec.num_q_heads,
                                          num_kv_heads=spec.num_kv_heads, sm_scale=spec.sm_scale,
                                          kv_dtype=1, k_scale=ks.cpu().numpy(),
                                          v_scale=vs.cpu().numpy(), nthreads=NTHREADS)
    sel = torch.from_numpy(rows).to(DEV)
    assert_close(out[sel], ref, "mixed-step prefill over e4m3")
    assert_lse_close(lse[sel], ref_lse, "mixed-step prefill over e4m3")
