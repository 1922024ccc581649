"""GPU parity of the short-query kernel (speculative verify, infer-lab
"Technique" table: at most 64 query rows = q_len x group per sequence), which
the ragged prefill entry takes when the host query lengths are given.  Each
case runs both kernels -- the short-query one (host lengths given) and the
tcgen05 prefill (no host lengths) -- against the oracle, over plans of one to
four KV chunks (clusters of 2-4 CTAs merge through distributed shared
memory)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close, pool_np, u16

pytestmark = pytest.mark.gpu


def _spec(hq, hkv, d, n, seed):
    return wl.PrefillSpec("short queries", num_chunks=n, chunk_len=4, prefix_lo=0, prefix_hi=100,
                          num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=seed)


def _run(spec, pb, host, causal=True, window=-1):
    desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=pb.k_cache.shape[0],
                         max_blocks_per_seq=pb.tables_host.shape[1])
    T = int(pb.qo_indptr_host[-1])
    out = torch.full((T, spec.num_q_heads, spec.head_dim), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, spec.num_q_heads), float("nan"), device=DEV)
    pkv.pkv_prefill_attention_ragged(
        desc, pb.q.to(DEV), torch.from_numpy(pb.qo_indptr_host).to(DEV), pb.k_cache.to(DEV),
        pb.v_cache.to(DEV), torch.from_numpy(pb.tables_host).to(DEV),
        torch.from_numpy(pb.kv_lens_host).to(DEV), spec.sm_scale, out, lse,
        qo_indptr_host=pb.qo_indptr_host if host else None,
        kv_lens_host=pb.kv_lens_host if host else None, causal=causal, window=window)
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    return out, lse


def _oracle(spec, pb, causal=True, window=-1):
    return oracle.paged_attention(q=u16(pb.q), k_cache=pool_np(pb.k_cache), v_cache=pool_np(pb.v_cache),
                                  block_tables=pb.tables_host, qo_indptr=pb.qo_indptr_host,
                                  kv_lens=pb.kv_lens_host, num_q_heads=spec.num_q_heads,
                                  num_kv_heads=spec.num_kv_heads, sm_scale=spec.sm_scale, causal=causal,
                                  window=window, nthreads=NTHREADS)


# (Hq, Hkv, D): groups of 4, 8, 1, 16 and 3 rows per query token
SHAPES = [(32, 8, 128), (16, 2, 128), (8, 8, 64), (16, 1, 64), (12, 4, 128)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
@pytest.mark.parametrize("seqs,long_prefix", [(12, 3000), (3, 8000), (40, 1200)])
def test_short_queries_both_kernels_match_the_oracle(hq, hkv, d, seqs, long_prefix):
    G = hq // hkv
    rng = np.random.default_rng(hq * 7 + d + seqs)
    qmax = 64 // G
    q_lens = [int(v) for v in rng.integers(1, qmax + 1, seqs)]
    q_lens[0] = qmax  # a full 64-row (or 16-row-tile multiple) sequence
    pair_prefix = rng.integers(0, long_prefix + 1, (seqs + 1) // 2)
    pair_prefix[-1] = long_prefix  # the batch generator shares a prefix within each pair
    prefixes = [int(v) for v in np.repeat(pair_prefix, 2)[:seqs]]
    spec = _spec(hq, hkv, d, seqs, seed=seqs + d)
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=q_lens, prefixes=prefixes)
    ref, ref_lse = _oracle(spec, pb)
    for host in (True, False):
        out, lse = _run(spec, pb, host)
        what = "%s, %d/%d/%d, %d seqs" % ("short-query" if host else "tcgen05", hq, hkv, d, seqs)
        assert_close(out, ref, what)
        assert_lse_close(lse, ref_lse, what)


@pytest.mark.parametrize("causal,window", [(False, -1), (True, 128), (True, 1), (True, 40),
                                           (False, 100)])
def test_short_query_masks(causal, window):
    spec = _spec(32, 8, 128, 6, seed=5)
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[16, 1, 7, 3, 16, 9], prefixes=[0, 0, 500, 500, 2100, 2100])
    ref, ref_lse = _oracle(spec, pb, causal=causal, window=window)
    out, lse = _run(spec, pb, True, causal=causal, window=window)
    assert_close(out, ref, "short-query causal=%s window=%d" % (causal, window))
    assert_lse_close(lse, ref_lse, "short-query masks")
