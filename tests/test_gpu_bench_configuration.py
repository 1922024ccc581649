"""The benchmark's own workloads in the launch configuration bench.py times:
steps captured in a CUDA graph and replayed, decode steps whose descriptor
carries PKV_DESC_PREFETCH_KV, the Llama-3-8B-shaped mixed step as the ragged
prefill followed by a decode that does not wait for it (PKV_DESC_INDEPENDENT),
the Qwen2.5-3B-shaped step rotating over four batches of one pool, and the
FP8 step's full-attention and window layers.

After the replays, sampled sequences are checked against the oracle: their
appended cache rows byte for byte, and the attention outputs (decode and
prefill) within the attention tolerance.  Replaying a step rewrites the same
slot with the same bytes, so the state after any number of replays is that of
one step."""
import numpy as np
import pytest
import torch

import bench
import oracle
from tests._cases import BS
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close, compact_pool, u16

pytestmark = pytest.mark.gpu


def _run(W, order, replays=2):
    """Eager steps, then the same steps captured in a graph and replayed."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in order:
            W.step(i)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in order:
            W.step(i)
    for _ in range(replays):
        g.replay()
    torch.cuda.synchronize()


def _sample(lens, rng, extra=2):
    return sorted(set([int(np.argmin(lens)), int(np.argmax(lens))] +
                      rng.choice(len(lens), size=extra, replace=False).tolist()))


def _check_decode(W, b, seqs, before, label, check_out=True, window=-1):
    spec = W.spec
    k0, v0, tabs = before
    lens = b.lens_host[seqs]
    fp8 = spec.kv_dtype == "fp8_e4m3"
    ks = None if b.k_scale is None else b.k_scale.cpu().numpy()
    vs = None if b.v_scale is None else b.v_scale.cpu().numpy()
    q_rot = oracle.append_rope(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                               head_dim=spec.head_dim, block_size=BS, kv_dtype=1 if fp8 else 0,
                               k_cache=k0, v_cache=v0, block_tables=tabs,
                               token_to_seq=np.arange(len(seqs), dtype=np.int32),
                               positions=(lens - 1).astype(np.int32), k_new=u16(b.k_new)[seqs],
                               v_new=u16(b.v_new)[seqs], q=u16(b.q)[seqs],
                               cos_sin=oracle.rope_table(spec.rope_theta, spec.head_dim, W.max_ctx),
                               k_scale=ks, v_scale=vs)
    k1, v1, _ = compact_pool(b.k_cache, b.v_cache, b.tables_host, seqs)
    assert np.array_equal(k1, k0) and np.array_equal(v1, v0), "%s: appended rows differ" % label
    if not check_out:
        return
    ref, ref_lse = oracle.paged_attention(q=q_rot, k_cache=k0, v_cache=v0, block_tables=tabs,
                                          qo_indptr=np.arange(len(seqs) + 1), kv_lens=lens,
                                          num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                          sm_scale=spec.sm_scale, window=window, kv_dtype=1 if fp8 else 0,
                                          k_scale=ks, v_scale=vs, nthreads=NTHREADS)
    idx = torch.tensor(seqs, device=DEV)
    assert_close(W.out[idx], ref, label)
    assert_lse_close(W.lse[idx], ref_lse, label)


def test_mixed_step_as_benchmarked():
    """Llama-3-8B-shaped mixed step: prefill, then the decode step with
    PKV_DESC_INDEPENDENT | PKV_DESC_PREFETCH_KV, graph-replayed."""
    W = bench.DecodeWorkload(4, DEV, 0)
    assert W.independent and W.prefetch and W.prefill is not None
    rng = np.random.default_rng(41)
    b = W.insts[0]
    seqs = _sample(b.lens_host, rng, extra=1)
    before = compact_pool(b.k_cache, b.v_cache, b.tables_host, seqs)
    _run(W, [0, 0])
    assert W.pkv.pkv_device_errors(reset=True) == 0
    _check_decode(W, W.insts[0], seqs, before, "mixed-step decode as benchmarked")

    # the prefill half: every row of the sequence with the shortest prefix,
    # the last 16 query tokens of the one with the longest
    P = W.prefill
    pb = P.pb
    s_lo, s_hi = int(np.argmin(pb.prefix_host)), int(np.argmax(pb.prefix_host))
    qo = pb.qo_indptr_host
    parts = [(qo[s_lo], qo[s_lo + 1]), (qo[s_hi + 1] - 16, qo[s_hi + 1])]
    rows = np.concatenate([np.arange(lo, hi) for lo, hi in parts])
    sub_qo = np.array([0, parts[0][1] - parts[0][0], rows.size], dtype=np.int32)
    k, v, tabs = compact_pool(pb.k_cache, pb.v_cache, pb.tables_host, [s_lo, s_hi])
    ref, ref_lse = oracle.paged_attention(q=u16(pb.q)[rows], k_cache=k, v_cache=v, block_tables=tabs,
                                          qo_indptr=sub_qo, kv_lens=pb.kv_lens_host[[s_lo, s_hi]],
                                          num_q_heads=P.spec.num_q_heads, num_kv_heads=P.spec.num_kv_heads,
                                          sm_scale=P.spec.sm_scale, nthreads=NTHREADS)
    assert_close(P.out[torch.from_numpy(rows).to(DEV)], ref, "mixed-step prefill as benchmarked")


def test_rotating_decode_step_as_benchmarked():
    """Qwen2.5-3B-shaped step over four batches of one pool, each step's
    predecessor the previous batch's step, with PKV_DESC_PREFETCH_KV."""
    W = bench.DecodeWorkload(2, DEV, 0)
    assert W.prefetch and W.n_inst == 4
    rng = np.random.default_rng(42)
    samples, befores = {}, {}
    for i in range(W.n_inst):
        b = W.insts[i]
        samples[i] = _sample(b.lens_host, rng)
        befores[i] = compact_pool(b.k_cache, b.v_cache, b.tables_host, samples[i])
    order = list(range(W.n_inst))
    _run(W, order, replays=3)
    assert W.pkv.pkv_device_errors(reset=True) == 0
    last = order[-1]
    for i in order:
        # the shared output buffer holds the last batch's result
        _check_decode(W, W.insts[i], samples[i], befores[i], "rotating step, batch %d" % i,
                      check_out=i == last)


def test_fp8_two_layer_step_as_benchmarked():
    """FP8 e4m3 step: a full-attention layer, then the window-128 layer (its
    own pools and scales), each launch's predecessor the other layer's,
    with PKV_DESC_PREFETCH_KV.  Both layers' appended rows are checked; the
    shared output buffer holds the window layer's result."""
    W = bench.DecodeWorkload(5, DEV, 0)
    assert W.prefetch and len(W.layers) == 2
    rng = np.random.default_rng(43)
    b0 = W.layers[0][0]
    seqs = _sample(b0.lens_host, rng)
    befores = [compact_pool(layer[0].k_cache, layer[0].v_cache, layer[0].tables_host, seqs)
               for layer in W.layers]
    _run(W, [0, 0])
    assert W.pkv.pkv_device_errors(reset=True) == 0
    for li, (layer, w) in enumerate(zip(W.layers, W.windows)):
        _check_decode(W, layer[0], seqs, befores[li], "FP8 step, layer %d (window %d)" % (li, w),
                      check_out=li == len(W.layers) - 1, window=w)
