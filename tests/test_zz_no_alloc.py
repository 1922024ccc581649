"""The decode entry point for callers that cannot allocate device memory.

pkv_decode_attention_static takes no workspace: it runs on the library's own
fixed device scratch array.  It exists for callers that may not call
cudaMalloc where they call the library (inside an allocator callback, under a
framework that owns the memory pool, or in a plugin given only its tensors).
Here it is called twice in a row through the C ABI, on two different batches
that share the one scratch array, and each result is compared with
pkv_decode_attention on a caller workspace, within the attention tolerance
the other decode tests use.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import DEV, MAX_ERR, MEAN_ERR, desc_for, gpu_decode, on_device

pytestmark = pytest.mark.gpu


def test_static_scratch_decode_matches_workspace_decode_twice_in_a_row():
    spec = wl.QWEN25_3B   # the full Qwen2.5-3B-shaped batch: split, so the scratch is used
    batches = wl.make_decode_instances(spec, 2, DEV)
    results = []
    for b in batches:
        d = on_device(b)
        desc = desc_for(spec, b.k_cache, b.tables_host)
        assert pkv.pkv_decode_workspace_size(desc, spec.batch, b.max_context_len) > 0
        ref, ref_lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), device=DEV)
        pkv.pkv_decode_attention_static(desc, d["q"], d["k_cache"], d["v_cache"],
                                        d["block_tables"], d["context_lens"], b.max_context_len,
                                        spec.sm_scale, out, lse)
        torch.cuda.synchronize()
        results.append((out, lse, ref, ref_lse))
    for out, lse, ref, ref_lse in results:
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= MAX_ERR and err.mean().item() <= MEAN_ERR
        assert (lse - ref_lse).abs().max().item() <= 2e-3
    assert pkv.pkv_device_errors() == 0


def test_static_scratch_rejects_a_batch_beyond_its_size():
    spec = wl.scaled(wl.QWEN25_3B, batch=64)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    big = 4096  # 4096 seqs x 2 heads x 256 splits of 8 heads: far beyond 16 MiB
    need = pkv.pkv_decode_workspace_size(desc, big, b.max_context_len, -1, 1)
    assert need > 16 << 20
    lens = torch.ones(big, dtype=torch.int32, device=DEV)
    q = torch.zeros((big, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((big, b.tables_host.shape[1]), dtype=torch.int32, device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_static(desc, q, d["k_cache"], d["v_cache"], tables, lens,
                                        b.max_context_len, spec.sm_scale, torch.empty_like(q),
                                        chunk_blocks=1)
    assert e.value.status == 3 and "static" in str(e.value)
