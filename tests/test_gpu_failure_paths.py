"""Failure handling of the attention kernels, on the GPU, without a fault.

Device checks: a block id outside the pool and a context length beyond the
host's bound are planted in decode and in prefill inputs.  The kernels clamp
the access to a valid one, set the matching PKV_DEVERR bit and finish; every
other sequence still matches the oracle.

Bounded waits (the fail-stop deadline of RustInfer's "Configuration" and the
bounded self-check of its "Status"): a test hook makes one pipeline wait of
the first CTA wait on a barrier that nothing arrives on, with a 20 ms limit.
The kernel must give up, drain the copies it issued, set
PKV_DEVERR_TIMEOUT, leave every merge ticket at zero and return; the states
it did not touch still match the oracle, and the next call is clean.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import (DEV, assert_close, assert_lse_close, desc_for, gpu_decode, on_device,
                        oracle_decode, pool_np, u16)
from tests.test_gpu_prefill import _gpu_prefill, _oracle_prefill, _small

pytestmark = pytest.mark.gpu

LIMIT_US = 20000


def _decode_case():
    spec = wl.scaled(wl.QWEN25_3B, batch=12, ctx_hi=2000)
    b = wl.make_decode_batch(spec, "cpu")
    return spec, b


def _splits(b, chunk):
    return -(-((b.max_context_len + 15) // 16) // chunk)


def test_decode_flags_a_bad_block_id_and_keeps_the_other_sequences_exact():
    spec, b = _decode_case()
    tables = b.tables_host.copy()
    bad_seq = 3
    tables[bad_seq, 2] = b.k_cache.shape[0] + 7          # outside the pool
    d = on_device(b)
    d["block_tables"] = torch.from_numpy(tables).to(DEV)
    desc = desc_for(spec, b.k_cache, tables)
    pkv.pkv_device_errors(reset=True)
    out, lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_BLOCK_ID
    keep = [s for s in range(spec.batch) if s != bad_seq]
    ref, ref_lse = oracle_decode(spec, u16(b.q), pool_np(b.k_cache), pool_np(b.v_cache),
                                 b.tables_host, b.lens_host)
    assert torch.isfinite(out.float()).all()
    assert_close(out[keep], ref[keep], "decode beside a bad block id")
    assert_lse_close(lse[keep], ref_lse[keep], "decode beside a bad block id")


def test_decode_flags_a_length_beyond_the_host_bound():
    spec, b = _decode_case()
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    long_seq = int(np.argmin(b.lens_host))
    lens = b.context_lens.clone()
    lens[long_seq] = b.max_context_len + 37              # the host bound says otherwise
    d["context_lens"] = lens.to(DEV)
    pkv.pkv_device_errors(reset=True)
    out, lse, ws = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_LENGTH
    keep = [s for s in range(spec.batch) if s != long_seq]
    ref, ref_lse = oracle_decode(spec, u16(b.q), pool_np(b.k_cache), pool_np(b.v_cache),
                                 b.tables_host, b.lens_host)
    assert_close(out[keep], ref[keep], "decode beside a length beyond the bound")
    assert_lse_close(lse[keep], ref_lse[keep], "decode beside a length beyond the bound")
    assert int(ws[:spec.batch * spec.num_kv_heads * 4].count_nonzero()) == 0


def test_prefill_flags_a_bad_block_id_and_a_length_beyond_the_table():
    spec = _small()
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[96, 80, 37, 130], prefixes=[300, 300, 515, 515])
    tables = pb.tables_host.copy()
    bad_id_seq, long_seq = 1, 2
    tables[bad_id_seq, 1] = pb.k_cache.shape[0] + 3
    kvl_dev = pb.kv_lens_host.copy()
    kvl_dev[long_seq] = tables.shape[1] * 16 + 50        # beyond the table; host copy is valid
    desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=pb.k_cache.shape[0],
                         max_blocks_per_seq=tables.shape[1])
    out = torch.full((pb.total_q, spec.num_q_heads, spec.head_dim), float("nan"),
                     dtype=torch.bfloat16, device=DEV)
    lse = torch.full((pb.total_q, spec.num_q_heads), float("nan"), device=DEV)
    pkv.pkv_device_errors(reset=True)
    pkv.pkv_prefill_attention_ragged(desc, pb.q.to(DEV), torch.from_numpy(pb.qo_indptr_host).to(DEV),
                                     pb.k_cache.to(DEV), pb.v_cache.to(DEV),
                                     torch.from_numpy(tables).to(DEV),
                                     torch.from_numpy(kvl_dev).to(DEV), spec.sm_scale, out, lse,
                                     qo_indptr_host=pb.qo_indptr_host,
                                     kv_lens_host=pb.kv_lens_host)
    torch.cuda.synchronize()
    flags = pkv.pkv_device_errors(reset=True)
    assert flags & pkv.DEVERR_BLOCK_ID and flags & pkv.DEVERR_LENGTH
    ref, ref_lse = _oracle_prefill(spec, pb)
    qo = pb.qo_indptr_host
    rows = np.concatenate([np.arange(qo[s], qo[s + 1]) for s in range(len(qo) - 1)
                           if s not in (bad_id_seq, long_seq)])
    assert_close(out[rows], ref[rows], "prefill beside planted bad inputs")
    assert_lse_close(lse[rows], ref_lse[rows], "prefill beside planted bad inputs")


@pytest.mark.parametrize("chunk", [4, 40])   # ticket merge (>4 chunks), cluster merge (2-4)
def test_decode_wait_timeout_gives_up_cleanly(chunk):
    spec, b = _decode_case()
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    n = _splits(b, chunk)
    assert (n > 4) if chunk == 4 else (2 <= n <= 4)
    ref, ref_lse = oracle_decode(spec, u16(b.q), pool_np(b.k_cache), pool_np(b.v_cache),
                                 b.tables_host, b.lens_host)
    pkv.pkv_device_errors(reset=True)
    pkv.pkv_test_inject_wait_timeout(1, LIMIT_US)
    try:
        out, lse, ws = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, chunk=chunk)
    finally:
        pkv.pkv_test_inject_wait_timeout(0)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_TIMEOUT
    assert int(ws[:spec.batch * spec.num_kv_heads * 4].count_nonzero()) == 0, \
        "tickets must be left at zero after a give-up"
    assert torch.isfinite(out.float()).all()
    G = spec.num_q_heads // spec.num_kv_heads
    # every state but the first CTA's (sequence 0, KV head 0) is untouched
    o, r = out.float().cpu().numpy(), ref.copy()
    o[0, :G] = r[0, :G] = 0.0
    assert_close(torch.from_numpy(o), r, "decode after a give-up (chunk %d)" % chunk)
    # the next call is clean
    out2, lse2, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, chunk=chunk)
    assert pkv.pkv_device_errors(reset=True) == 0
    assert_close(out2, ref, "decode after the hook is disarmed")
    assert_lse_close(lse2, ref_lse, "decode after the hook is disarmed")


def test_prefill_wait_timeout_gives_up_cleanly():
    spec = _small()
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[96, 1, 37, 130], prefixes=[0, 0, 515, 515])
    ref, ref_lse = _oracle_prefill(spec, pb)
    pkv.pkv_device_errors(reset=True)
    pkv.pkv_test_inject_wait_timeout(2, LIMIT_US)
    try:
        out, lse = _gpu_prefill(spec, pb)
    finally:
        pkv.pkv_test_inject_wait_timeout(0)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_TIMEOUT
    G = spec.num_q_heads // spec.num_kv_heads
    # the first CTA serves KV head 0 only: every other head is untouched, and
    # the tile that gave up wrote finite values (zeros)
    assert torch.isfinite(out.float()).all()
    assert_close(out[:, G:], ref[:, G:], "prefill after a give-up")
    assert_lse_close(lse[:, G:], ref_lse[:, G:], "prefill after a give-up")
    out2, lse2 = _gpu_prefill(spec, pb)
    assert pkv.pkv_device_errors(reset=True) == 0
    assert_close(out2, ref, "prefill after the hook is disarmed")
    assert_lse_close(lse2, ref_lse, "prefill after the hook is disarmed")


def test_fp8_prefill_wait_timeout_gives_up_cleanly():
    """The same give-up over e4m3 pools: the producers convert code slots in
    shared memory, so their drain (every code load issued, and Q) and the
    softmax warps' Q conversion take part in it."""
    import oracle
    from tests._gpu import NTHREADS, u8
    spec = _small()
    pb = wl.make_prefill_batch(spec, "cpu", q_lens=[96, 1, 37, 130], prefixes=[0, 0, 515, 515])
    ks = (pb.k_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
    vs = (pb.v_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
    k8 = (pb.k_cache.float() / ks.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (pb.v_cache.float() / vs.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                         head_dim=spec.head_dim, num_blocks=k8.shape[0],
                         max_blocks_per_seq=pb.tables_host.shape[1], kv_dtype=pkv.KV_FP8_E4M3)
    ref, ref_lse = oracle.paged_attention(
        q=u16(pb.q), k_cache=u8(k8), v_cache=u8(v8), block_tables=pb.tables_host,
        qo_indptr=pb.qo_indptr_host, kv_lens=pb.kv_lens_host, num_q_heads=spec.num_q_heads,
        num_kv_heads=spec.num_kv_heads, sm_scale=spec.sm_scale, kv_dtype=1, k_scale=ks.numpy(),
        v_scale=vs.numpy(), nthreads=NTHREADS)

    def call():
        out = torch.full((pb.total_q, spec.num_q_heads, spec.head_dim), float("nan"),
                         dtype=torch.bfloat16, device=DEV)
        lse = torch.full((pb.total_q, spec.num_q_heads), float("nan"), device=DEV)
        pkv.pkv_prefill_attention_ragged(desc, pb.q.to(DEV), torch.from_numpy(pb.qo_indptr_host).to(DEV),
                                         k8.to(DEV), v8.to(DEV), torch.from_numpy(pb.tables_host).to(DEV),
                                         torch.from_numpy(pb.kv_lens_host).to(DEV), spec.sm_scale, out, lse,
                                         qo_indptr_host=pb.qo_indptr_host, kv_lens_host=pb.kv_lens_host,
                                         k_scale=ks.to(DEV), v_scale=vs.to(DEV))
        torch.cuda.synchronize()
        return out, lse

    pkv.pkv_device_errors(reset=True)
    pkv.pkv_test_inject_wait_timeout(2, LIMIT_US)
    try:
        out, lse = call()
    finally:
        pkv.pkv_test_inject_wait_timeout(0)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_TIMEOUT
    G = spec.num_q_heads // spec.num_kv_heads
    assert torch.isfinite(out.float()).all()
    assert_close(out[:, G:], ref[:, G:], "e4m3 prefill after a give-up")
    assert_lse_close(lse[:, G:], ref_lse[:, G:], "e4m3 prefill after a give-up")
    out2, lse2 = call()
    assert pkv.pkv_device_errors(reset=True) == 0
    assert_close(out2, ref, "e4m3 prefill after the hook is disarmed")
    assert_lse_close(lse2, ref_lse, "e4m3 prefill after the hook is disarmed")
