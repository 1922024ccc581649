"""GPU parity of split-KV GQA decode against the oracle, element by element,
within max|err| <= 1e-2 and mean|err| <= 1e-3 (bf16 inputs, fp32
accumulation); plus the invariants the pages state (any split count, any
block placement, poisoned unused slots) and the full-size workloads on
sampled sequences."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import (DEV, NTHREADS, assert_close, assert_lse_close, compact_pool, desc_for,
                        gpu_decode, on_device, oracle_decode, pool_np, u16)

pytestmark = pytest.mark.gpu


def _scales(b):
    if b.k_scale is None:
        return None, None
    return b.k_scale.cpu().numpy(), b.v_scale.cpu().numpy()


def _check_batch(spec, b, d, window=-1, chunks=(0,)):
    desc = desc_for(spec, b.k_cache, b.tables_host)
    ks, vs = _scales(b)
    ref, ref_lse = oracle_decode(spec, u16(b.q), pool_np(b.k_cache), pool_np(b.v_cache),
                                 b.tables_host, b.lens_host, window, ks, vs)
    for chunk in chunks:
        out, lse, ws = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, window, chunk)
        # window 1: every output is one value row, so the literal figures
        # measure the bf16 rounding of O(1) values alone (~1.2e-3 mean)
        assert_close(out, ref, "%s chunk=%d window=%d" % (spec.name, chunk, window),
                     literal=window != 1)
        assert_lse_close(lse, ref_lse, spec.name)
        assert int(ws[:b.lens_host.size * spec.num_kv_heads * 4].count_nonzero()) == 0, \
            "ticket counters must be left at zero"
    assert pkv.pkv_device_errors() == 0


def test_tiny_workload_every_split_count():
    spec = wl.TINY
    b = wl.make_decode_batch(spec, "cpu")
    _check_batch(spec, b, on_device(b), chunks=(0, 1, 2, 3, 4, 7, 16, 128))


@pytest.mark.parametrize("cfg,batch,ctx_hi", [(2, 9, 4096), (3, 40, 768), (4, 5, 6000),
                                              (5, 7, 5000)])
def test_workload_shapes_reduced(cfg, batch, ctx_hi):
    spec = wl.scaled(wl.CONFIGS[cfg], batch=batch, ctx_hi=ctx_hi)
    b = wl.make_decode_batch(spec, "cpu")
    # bf16 pools take chunks of up to 256 blocks: past 128 a warp's blocks
    # 32-63 sit in each lane's second block-id register
    longer = (129, 200, 256) if spec.kv_dtype == "bf16" else ()
    _check_batch(spec, b, on_device(b), chunks=(0, 1, 5, 16, 128) + longer)


@pytest.mark.parametrize("fp8", [False, True])
def test_sliding_window(fp8):
    spec = wl.scaled(wl.FP8_DECODE if fp8 else wl.QWEN25_3B, batch=10, ctx_hi=3000)
    spec = wl.dataclasses.replace(spec, ctx_lo=1)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    for window in (128, 1, 17, 5000):
        _check_batch(spec, b, d, window=window, chunks=(0, 1, 3))


def test_odd_groups_and_lengths():
    # G = 1, 3, 5, 16; lengths 1..40 around block edges
    for hq, hkv, D in ((4, 4, 128), (6, 2, 64), (10, 2, 128), (32, 2, 64)):
        spec = wl.DecodeSpec("odd", batch=40, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                             ctx_lo=1, ctx_hi=40, seed=11, fixed_lens=tuple(range(1, 41)),
                             pool_blocks=200)
        b = wl.make_decode_batch(spec, "cpu")
        _check_batch(spec, b, on_device(b), chunks=(0, 1, 2))


@pytest.mark.parametrize("lens", [(1,), (16,) * 512, (5, 700, 16, 17, 1, 300, 33, 4000),
                                  tuple(range(1, 514))])
def test_automatic_plan_edges(lens):
    """Batches at the edges of the automatic split plan: a single key, 512
    one-block sequences, a mix of very short and long contexts, and 513
    sequences of every length from 1 to 513."""
    import dataclasses
    spec = dataclasses.replace(wl.scaled(wl.QWEN25_3B, batch=len(lens)), fixed_lens=lens,
                               ctx_lo=min(lens), ctx_hi=max(lens), seed=77)
    b = wl.make_decode_batch(spec, "cpu")
    _check_batch(spec, b, on_device(b), chunks=(0,))


def test_sequence_without_keys():
    """A sequence whose device-side length is 0 gets o = 0 and lse = -inf;
    the others are unchanged."""
    spec = wl.scaled(wl.QWEN3_4B, batch=9, ctx_hi=600, seed=5)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    ks, vs = _scales(b)
    lens = b.lens_host.copy()
    lens[3] = 0
    d["context_lens"] = torch.from_numpy(lens).to(DEV)
    out, lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
    keep = [i for i in range(len(lens)) if i != 3]
    ref, ref_lse = oracle_decode(spec, u16(b.q[keep]), pool_np(b.k_cache), pool_np(b.v_cache),
                                 b.tables_host[keep], b.lens_host[keep])
    assert_close(out[keep], ref, "other sequences")
    assert_lse_close(lse[keep], ref_lse, "other sequences")
    assert torch.count_nonzero(out[3].float()).item() == 0
    assert bool(torch.all(torch.isinf(lse[3]) & (lse[3] < 0)))
    assert pkv.pkv_device_errors() == 0


def test_poisoned_unused_slots_do_not_change_the_output():
    spec = wl.scaled(wl.QWEN25_3B, batch=6, ctx_hi=700)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    out1, lse1, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, chunk=2)
    # NaN in every slot no sequence can see: tail rows of last blocks, unused blocks
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    used = np.zeros((kc.shape[0], 16), bool)
    for s, n in enumerate(b.lens_host):
        for t in range(n):
            used[b.tables_host[s, t // 16], t % 16] = True
    mask = torch.from_numpy(~used).to(DEV)[:, None, :, None].expand_as(kc)
    kc[mask] = float("nan")
    vc[mask] = float("nan")
    d2 = dict(d, k_cache=kc, v_cache=vc)
    for chunk in (0, 2):
        out2, lse2, _ = gpu_decode(desc, d2, b.max_context_len, spec.sm_scale, chunk=chunk)
        if chunk == 2:
            assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
        assert torch.isfinite(out2.float()).all()


def test_block_placement_and_split_count_invariance():
    spec = wl.scaled(wl.QWEN3_4B, batch=16, ctx_hi=768)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    out1, _, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, chunk=4)
    perm = torch.randperm(b.k_cache.shape[0], generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)
    d2 = dict(d, k_cache=d["k_cache"][perm.to(DEV)].contiguous(),
              v_cache=d["v_cache"][perm.to(DEV)].contiguous())
    tabs = d["block_tables"].long()
    d2["block_tables"] = torch.where(tabs >= 0, inv.to(DEV)[tabs.clamp(min=0)], -1).to(torch.int32)
    out2, _, _ = gpu_decode(desc, d2, b.max_context_len, spec.sm_scale, chunk=4)
    assert torch.equal(out1, out2)  # same bytes, same order of arithmetic


def test_decode_after_append_qwen3_4b_full_size():
    """The Qwen3-4B-shaped workload end to end: append the new token with
    RoPE (theta 1e6) at ctx-1, then decode -- both sides from the same seeded
    bytes, the oracle doing its own append."""
    spec = wl.QWEN3_4B
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    table = pkv.pkv_rope_cos_sin_table(spec.rope_theta, spec.head_dim, int(b.lens_host.max()))
    seq = torch.arange(spec.batch, dtype=torch.int32, device=DEV)
    pos = (d["context_lens"] - 1).to(torch.int32)
    pkv.pkv_append_rope(desc, d["k_cache"], d["v_cache"], d["block_tables"], seq, pos,
                        d["k_new"], d["v_new"], q=d["q"], cos_sin=torch.from_numpy(table).to(DEV))
    out, lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale)
    kh, vh = pool_np(b.k_cache).copy(), pool_np(b.v_cache).copy()
    qh = oracle.append_rope(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                            head_dim=spec.head_dim, block_size=16, kv_dtype=0, k_cache=kh,
                            v_cache=vh, block_tables=b.tables_host,
                            token_to_seq=np.arange(spec.batch), positions=b.lens_host - 1,
                            k_new=u16(b.k_new), v_new=u16(b.v_new), q=u16(b.q),
                            cos_sin=oracle.rope_table(spec.rope_theta, spec.head_dim,
                                                      int(b.lens_host.max())))
    assert np.array_equal(u16(d["q"]), qh)
    ref, ref_lse = oracle_decode(spec, qh, kh, vh, b.tables_host, b.lens_host)
    assert_close(out, ref, "Qwen3-4B full")
    assert_lse_close(lse, ref_lse, "Qwen3-4B full")


@pytest.mark.parametrize("cfg,window", [(2, -1), (4, -1), (5, -1), (5, wl.FP8_WINDOW)])
def test_full_size_workloads_on_sampled_sequences(cfg, window):
    """The full-size batches, in the launch configuration the benchmark uses
    (planned split), generated on the GPU; a sample of sequences (shortest,
    longest, and random ones) is checked element by element against the
    oracle on a host copy of just their blocks."""
    spec = wl.CONFIGS[cfg]
    b = wl.make_decode_batch(spec, DEV)
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    out, lse, _ = gpu_decode(desc, d, b.max_context_len, spec.sm_scale, window)
    rng = np.random.default_rng(cfg)
    seqs = sorted(set([int(np.argmin(b.lens_host)), int(np.argmax(b.lens_host))] +
                      rng.choice(spec.batch, size=4, replace=False).tolist()))
    k, v, tabs = compact_pool(b.k_cache, b.v_cache, b.tables_host, seqs)
    ks, vs = _scales(b)
    ref, ref_lse = oracle_decode(spec, u16(b.q)[seqs], k, v, tabs, b.lens_host[seqs], window, ks,
                                 vs)
    assert_close(out[seqs], ref, "%s sampled" % spec.name)
    assert_lse_close(lse[seqs], ref_lse, spec.name)
    assert pkv.pkv_device_errors() == 0
