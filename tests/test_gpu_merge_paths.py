"""GPU parity of the two ways split-KV decode merges its chunks (FlashAttention-2
work partitioning, cited under llm-infer "References"): plans of 2..4 chunks
per sequence merge inside a thread-block cluster through distributed shared
memory, larger plans through the workspace and a ticket.  Every plan must
match the oracle, with and without sink logits, for bf16 and e4m3 pools."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from tests._cases import PagedCase
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

# 64 blocks at most: chunk c gives ceil(64 / c) chunks for the longest sequence
CHUNKS = {64: 1, 32: 2, 22: 3, 16: 4, 13: 5, 11: 6, 10: 7, 8: 8, 7: 10, 4: 16}

# (Hq, Hkv, D, e4m3): both head dims, both pool types, group sizes 4..8
SHAPES = [(16, 2, 128, False), (64, 8, 64, True), (16, 4, 64, False), (32, 8, 128, True),
          (16, 4, 64, True), (16, 2, 64, True)]


def _pool(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if bits.dtype == np.uint16:
        return t.view(torch.int16).view(torch.bfloat16).to(DEV)
    return t.to(DEV)


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("hq,hkv,d,fp8", SHAPES)
def test_cluster_and_ticket_merges_match_the_oracle(hq, hkv, d, fp8):
    rng = np.random.default_rng(120 + hq + hkv + d + fp8)
    lens = [1, 16, 17, 100, 257, 511, 700, 1024]
    case = PagedCase(rng, lens, hq, hkv, d, fp8=fp8)
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=case.num_blocks,
                         max_blocks_per_seq=case.mbps, kv_dtype=1 if fp8 else 0)
    B = len(lens)
    max_ctx = max(lens)
    sinks = rng.uniform(-1.0, 5.0, hq).astype(np.float32)
    kd, vd, q = _pool(case.k_cache), _pool(case.v_cache), _pool(case.q)
    tabs, lens_d = _dev(case.tables), _dev(case.lens)
    ks, vs = _dev(case.k_scale), _dev(case.v_scale)
    for sk in (None, sinks):
        ref, ref_lse = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=1 / math.sqrt(d),
                                              sinks=sk, nthreads=NTHREADS)
        for chunk, splits in CHUNKS.items():
            assert -(-((max_ctx + 15) // 16) // chunk) == splits
            ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, chunk), 256),
                             dtype=torch.uint8, device=DEV)
            out = torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
            lse = torch.full((B, hq), float("nan"), device=DEV)
            pkv.pkv_decode_attention(desc, q, kd, vd, tabs, lens_d, max_ctx, 1 / math.sqrt(d), out, lse,
                                     ws, chunk_blocks=chunk, k_scale=ks, v_scale=vs, sinks=_dev(sk))
            torch.cuda.synchronize()
            what = "%s, %d chunks%s" % ("e4m3" if fp8 else "bf16", splits, ", sinks" if sk is not None else "")
            assert_close(out, ref, what)
            assert_lse_close(lse, ref_lse, what)
            assert int(ws[:4 * B * hkv].count_nonzero()) == 0, "tickets not reset"
    assert pkv.pkv_device_errors() == 0
