"""GPU parity of split-KV decode on ragged batches at the planner's edges
(FlashAttention-2 work partitioning, llm-infer "References"): long and
one-block sequences mixed, sequences without keys at the batch's ends, a
batch with fewer blocks than the GPU has CTA slots, sink logits on groups of
1 to 16 heads, and 400 short sequences.

Each case runs the automatic plan (chunk_blocks = 0: 2-4 chunks merged in a
thread-block cluster on these shapes) and a 4-block chunk (up to 64 chunks
per sequence, merged through the workspace ticket) on the same bytes, checks
both against the oracle, and that the tickets are left at zero."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from tests._cases import PagedCase
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _pool(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.int16).view(torch.bfloat16).to(DEV)


def _run(case, chunk, sinks=None):
    B = len(case.lens)
    desc = pkv.make_desc(num_q_heads=case.hq, num_kv_heads=case.hkv, head_dim=case.d,
                         num_blocks=case.k_cache.shape[0], max_blocks_per_seq=case.tables.shape[1])
    max_ctx = max(int(case.lens.max()), 1)
    ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, chunk), 256),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((B, case.hq, case.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, case.hq), float("nan"), device=DEV)
    pkv.pkv_decode_attention(desc, _pool(case.q), _pool(case.k_cache), _pool(case.v_cache),
                             _dev(case.tables), _dev(case.lens), max_ctx, 1 / math.sqrt(case.d), out, lse,
                             ws, chunk_blocks=chunk, sinks=_dev(sinks))
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    assert int(ws[:4 * B * case.hkv].count_nonzero()) == 0, "tickets not reset"
    return desc, out, lse


def _oracle(case, sinks=None):
    B = len(case.lens)
    return oracle.paged_attention(q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                                  block_tables=case.tables, qo_indptr=np.arange(B + 1), kv_lens=case.lens,
                                  num_q_heads=case.hq, num_kv_heads=case.hkv,
                                  sm_scale=1 / math.sqrt(case.d), sinks=sinks, nthreads=NTHREADS)


def _check(case, what, sinks=None):
    ref, ref_lse = _oracle(case, sinks)
    for chunk in (0, 4):
        _, out, lse = _run(case, chunk, sinks)
        assert_close(out, ref, "chunk_blocks=%d, %s" % (chunk, what))
        assert_lse_close(lse, ref_lse, "chunk_blocks=%d, %s" % (chunk, what))


# (Hq, Hkv, D): groups of 8, 4, 1, 16, 3 and 16 with one KV head
SHAPES = [(16, 2, 128), (32, 8, 128), (8, 8, 64), (32, 2, 64), (12, 4, 128), (16, 1, 128)]


@pytest.mark.parametrize("hq,hkv,d", SHAPES)
def test_ragged_batch(hq, hkv, d):
    rng = np.random.default_rng(hq * 31 + hkv + d)
    lens = rng.integers(1, 3000, 24)
    lens[:6] = [1, 15, 16, 17, 4096, 600]
    _check(PagedCase(rng, lens, hq, hkv, d), "%d/%d/%d" % (hq, hkv, d))


def test_zero_length_sequences_at_the_ends():
    """Sequences without keys -- first, last and in runs -- get o = 0 and
    lse = -inf; the others are unchanged."""
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 2500, 24)
    lens[[0, 5, 6, 7, 23]] = 0
    case = PagedCase(rng, np.maximum(lens, 1), 16, 2, 128)
    case.lens = lens.astype(np.int32)  # the cache holds a block for each, unused
    keep = [i for i in range(len(lens)) if lens[i] > 0]
    ref, ref_lse = oracle.paged_attention(q=case.q[keep], k_cache=case.k_cache, v_cache=case.v_cache,
                                          block_tables=case.tables[keep], qo_indptr=np.arange(len(keep) + 1),
                                          kv_lens=case.lens[keep], num_q_heads=16, num_kv_heads=2,
                                          sm_scale=1 / math.sqrt(128), nthreads=NTHREADS)
    for chunk in (0, 4):
        _, out, lse = _run(case, chunk)
        assert_close(out[keep], ref, "with empty sequences, chunk_blocks=%d" % chunk)
        assert_lse_close(lse[keep], ref_lse, "with empty sequences")
        empty = [i for i in range(len(lens)) if lens[i] == 0]
        assert torch.count_nonzero(out[empty].float()).item() == 0
        assert bool(torch.all(torch.isinf(lse[empty]) & (lse[empty] < 0)))


@pytest.mark.parametrize("lens", [(600,), (530, 530), (1, 1, 700)])
def test_fewer_blocks_than_cta_slots(lens):
    """Tiny batches: a few CTAs, each sequence cut into 2 chunks (or 38 of 4 blocks)."""
    rng = np.random.default_rng(len(lens))
    _check(PagedCase(rng, lens, 32, 8, 128), "tiny %s" % (lens,))


def test_sinks_on_whole_and_merged_sequences():
    rng = np.random.default_rng(9)
    lens = rng.integers(1, 2000, 40)
    lens[:3] = [3, 20, 4000]
    case = PagedCase(rng, lens, 16, 2, 128)
    sinks = rng.standard_normal(16).astype(np.float32) * 2
    _check(case, "sinks", sinks=sinks)


def test_large_batch_of_short_sequences():
    """400 one-head sequences (D = 64, G = 8) of 1 to 2000 keys."""
    rng = np.random.default_rng(400)
    lens = rng.integers(1, 2000, 400)
    lens[0] = 2000
    _check(PagedCase(rng, lens, 8, 1, 64), "B=400")
