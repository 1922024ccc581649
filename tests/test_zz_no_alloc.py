"""The decode entry point for callers that cannot allocate device memory.

pkv_decode_attention_static takes no workspace: it runs on the library's own
fixed device scratch array.  It exists for callers that may not call
cudaMalloc where they call the library (inside an allocator callback, under a
framework that owns the memory pool, or in a plugin given only its tensors).

The calls below force plans of more than four chunks per (sequence, KV head),
so the kernel writes its partial states into the static array and merges them
through tickets kept there -- the path that depends on the array.  Three
calls in a row use different batch sizes and chunk lengths: the second
call's tickets sit where the first call left partial states, so a ticket
that was not cleared would corrupt its merge.  Each result is compared
element by element with the oracle, within the attention tolerance of the
other decode tests, and bit for bit with pkv_decode_attention on a caller
workspace (the same kernel and plan).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import (DEV, assert_close, assert_lse_close, compact_pool, desc_for, gpu_decode,
                        on_device, oracle_decode, u16)

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


def _static_call(desc, d, max_ctx, sm_scale, chunk):
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    pkv.pkv_decode_attention_static(desc, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                    d["context_lens"], max_ctx, sm_scale, out, lse,
                                    chunk_blocks=chunk)
    return out, lse


def test_static_scratch_ticket_merges_match_oracle_three_calls_in_a_row():
    # (batch, chunk): fewer pairs first, so the second call's tickets land on
    # the first call's partial states in the shared array
    plans = [(32, 16), (64, 24), (32, 16)]
    batches = {n: wl.make_decode_batch(wl.scaled(wl.QWEN25_3B, batch=n), "cpu") for n in (32, 64)}
    results = []
    for n, chunk in plans:
        spec = wl.scaled(wl.QWEN25_3B, batch=n)
        b = batches[n]
        d = on_device(b)
        desc = desc_for(spec, b.k_cache, b.tables_host)
        max_blocks = (b.max_context_len + 15) // 16
        assert (max_blocks + chunk - 1) // chunk > 4, "the plan must merge through tickets"
        need = pkv.pkv_decode_workspace_size(desc, n, b.max_context_len, -1, chunk)
        assert 0 < need <= STATIC_BYTES
        out, lse = _static_call(desc, d, b.max_context_len, spec.sm_scale, chunk)
        torch.cuda.synchronize()
        ref_out, ref_lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, chunk=chunk)
        results.append((spec, b, out.clone(), lse.clone(), ref_out, ref_lse))
    for spec, b, out, lse, ref_out, ref_lse in results:
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), \
            "static scratch and caller workspace differ on the same plan"
        seqs = list(range(spec.batch))
        k, v, tabs = compact_pool(b.k_cache, b.v_cache, b.tables_host, seqs)
        ref, rl = oracle_decode(spec, u16(b.q), k, v, tabs, b.lens_host)
        assert_close(out, ref, "static scratch, batch %d" % spec.batch)
        assert_lse_close(lse, rl, "static scratch, batch %d" % spec.batch)
    assert pkv.pkv_device_errors() == 0


def test_static_scratch_rejects_a_batch_beyond_its_size():
    spec = wl.scaled(wl.QWEN25_3B, batch=64)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    big = 4096  # 4096 seqs x 2 heads x 256 splits of 8 heads: far beyond 16 MiB
    need = pkv.pkv_decode_workspace_size(desc, big, b.max_context_len, -1, 1)
    assert need > STATIC_BYTES
    lens = torch.ones(big, dtype=torch.int32, device=DEV)
    q = torch.zeros((big, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((big, b.tables_host.shape[1]), dtype=torch.int32, device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_static(desc, q, d["k_cache"], d["v_cache"], tables, lens,
                                        b.max_context_len, spec.sm_scale, torch.empty_like(q),
                                        chunk_blocks=1)
    assert e.value.status == 3 and "static" in str(e.value)
