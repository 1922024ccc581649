"""GPU parity of the ragged prefill over a sliding-window ring cache with its
cache commit (RustInfer, "Status": Tensor Core prefill over chunked inputs
followed by a stream-ordered cache commit; SWA with a 128-token ring cache).

The reference is the oracle's attention over a *linear* cache that holds
every sequence in full, its chunk appended by the oracle's own append (the
e4m3 quantisation included): ring == linear.  Chunks longer than the ring,
chunks of one token and empty prefixes are covered, through both the
short-query kernel (few query rows) and the tcgen05 kernel.  After the call
the ring must hold, byte for byte, the window of every sequence as the
linear cache holds it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from tests._cases import BS, bf16_bits, e4m3_codes
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

WINDOW = 128
RING = (WINDOW - 1 + BS - 1) // BS + 1   # 9 blocks hold any 128-key window


def _build(rng, prefixes, q_lens, hq, hkv, d, fp8):
    prefixes = np.asarray(prefixes, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    kv = prefixes + q_lens
    B = len(kv)
    nblk = (kv + BS - 1) // BS
    mbps = int(max(nblk.max(), RING))
    nb = int(nblk.sum()) + 8
    perm = rng.permutation(nb).astype(np.int32)
    lin_tab = np.full((B, mbps), -1, np.int32)
    off = 0
    for s in range(B):
        lin_tab[s, :nblk[s]] = perm[off:off + nblk[s]]
        off += nblk[s]
    if fp8:
        k_scale = (0.02 + 0.01 * np.arange(hkv)).astype(np.float32)
        v_scale = (0.03 + 0.01 * np.arange(hkv)).astype(np.float32)
        k_lin = e4m3_codes(rng.standard_normal((nb, hkv, BS, d)) / k_scale[None, :, None, None])
        v_lin = e4m3_codes(rng.standard_normal((nb, hkv, BS, d)) / v_scale[None, :, None, None])
    else:
        k_scale = v_scale = None
        k_lin = bf16_bits(rng.standard_normal((nb, hkv, BS, d)))
        v_lin = bf16_bits(rng.standard_normal((nb, hkv, BS, d)))
    T = int(q_lens.sum())
    k_chunk = bf16_bits(rng.standard_normal((T, hkv, d)))
    v_chunk = bf16_bits(rng.standard_normal((T, hkv, d)))
    qo = np.zeros(B + 1, np.int32)
    qo[1:] = np.cumsum(q_lens)
    # the ring holds each sequence's last RING prefix blocks (what the appends left)
    k_ring = np.zeros((B * RING + 3, hkv, BS, d), k_lin.dtype)
    v_ring = np.zeros_like(k_ring)
    ring_perm = rng.permutation(B * RING + 3).astype(np.int32)
    ring_tab = np.full((B, mbps), -1, np.int32)
    for s in range(B):
        ring_tab[s, :RING] = ring_perm[s * RING:(s + 1) * RING]
        for b in range((int(prefixes[s]) + BS - 1) // BS):
            k_ring[ring_tab[s, b % RING]] = k_lin[lin_tab[s, b]]
            v_ring[ring_tab[s, b % RING]] = v_lin[lin_tab[s, b]]
    # the linear reference: the chunk appended by the oracle's own append
    tts = np.repeat(np.arange(B), q_lens).astype(np.int32)
    pos = np.concatenate([np.arange(prefixes[s], kv[s]) for s in range(B)]).astype(np.int32)
    oracle.append_rope(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS,
                       kv_dtype=1 if fp8 else 0, k_cache=k_lin, v_cache=v_lin, block_tables=lin_tab,
                       token_to_seq=tts, positions=pos, k_new=k_chunk, v_new=v_chunk,
                       k_scale=k_scale, v_scale=v_scale)
    q = bf16_bits(rng.standard_normal((T, hq, d)))
    return dict(kv=kv, qo=qo, q=q, k_lin=k_lin, v_lin=v_lin, lin_tab=lin_tab, k_ring=k_ring,
                v_ring=v_ring, ring_tab=ring_tab, k_chunk=k_chunk, v_chunk=v_chunk,
                k_scale=k_scale, v_scale=v_scale, hq=hq, hkv=hkv, d=d, fp8=fp8)


def _t(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(DEV)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("prefixes,q_lens", [([0, 100, 1000, 5], [1, 7, 3, 2]),
                                             ([0, 100, 1000, 5], [300, 1, 40, 130]),
                                             ([2000, 37], [517, 200])])
def test_ring_prefill_equals_linear_and_commits_the_window(fp8, prefixes, q_lens):
    rng = np.random.default_rng(sum(q_lens) + len(prefixes) + 7 * fp8)
    hq, hkv, d = (64, 8, 64) if fp8 else (16, 4, 128)
    c = _build(rng, prefixes, q_lens, hq, hkv, d, fp8)
    sm_scale = 1.0 / math.sqrt(d)
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                         num_blocks=c["k_ring"].shape[0], max_blocks_per_seq=c["ring_tab"].shape[1],
                         kv_dtype=1 if fp8 else 0, ring_blocks=RING)
    T = int(c["qo"][-1])
    ws = torch.empty(pkv.pkv_prefill_ring_workspace_size(desc, len(c["kv"]), WINDOW, max(q_lens)),
                     dtype=torch.uint8, device=DEV)
    kr, vr = _t(c["k_ring"]), _t(c["v_ring"])
    out = torch.full((T, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, hq), float("nan"), device=DEV)
    ks = None if c["k_scale"] is None else _t(c["k_scale"])
    vs = None if c["v_scale"] is None else _t(c["v_scale"])
    pkv.pkv_device_errors(reset=True)
    pkv.pkv_prefill_ring_commit(desc, _t(c["q"]), _t(c["qo"]), _t(c["k_chunk"]), _t(c["v_chunk"]),
                                kr, vr, _t(c["ring_tab"]), _t(c["kv"]), sm_scale, WINDOW, out,
                                c["qo"], c["kv"], ws, lse=lse, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkv.pkv_device_errors() == 0
    ref, ref_lse = oracle.paged_attention(
        q=c["q"], k_cache=c["k_lin"], v_cache=c["v_lin"], block_tables=c["lin_tab"],
        qo_indptr=c["qo"], kv_lens=c["kv"], num_q_heads=hq, num_kv_heads=hkv, sm_scale=sm_scale,
        causal=True, window=WINDOW, kv_dtype=1 if fp8 else 0, k_scale=c["k_scale"],
        v_scale=c["v_scale"], nthreads=NTHREADS)
    what = "ring prefill %s q=%s" % ("e4m3" if fp8 else "bf16", q_lens)
    assert_close(out, ref, what, literal=min(prefixes) > 0)   # position 0 attends one key
    assert_lse_close(lse, ref_lse, what)
    # the commit: every position of each sequence's last window sits in its ring slot
    kr_h = kr.cpu().view(torch.uint8 if fp8 else torch.int16).numpy()
    vr_h = vr.cpu().view(torch.uint8 if fp8 else torch.int16).numpy()
    kl = c["k_lin"].view(np.uint8 if fp8 else np.int16)
    vl = c["v_lin"].view(np.uint8 if fp8 else np.int16)
    for s, n in enumerate(c["kv"]):
        for p in range(max(0, int(n) - WINDOW), int(n)):
            rb, lb = c["ring_tab"][s, (p // BS) % RING], c["lin_tab"][s, p // BS]
            assert np.array_equal(kr_h[rb, :, p % BS], kl[lb, :, p % BS]), (s, p)
            assert np.array_equal(vr_h[rb, :, p % BS], vl[lb, :, p % BS]), (s, p)


def test_ring_prefill_rejects_a_linear_desc_and_a_window_beyond_the_ring():
    rng = np.random.default_rng(3)
    c = _build(rng, [50], [20], 16, 4, 128, False)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    out = torch.empty((20, 16, 128), dtype=torch.bfloat16, device=DEV)
    for ring, window in ((0, WINDOW), (RING, 1000)):
        desc = pkv.make_desc(num_q_heads=16, num_kv_heads=4, head_dim=128,
                             num_blocks=c["k_ring"].shape[0],
                             max_blocks_per_seq=c["ring_tab"].shape[1], ring_blocks=ring)
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_prefill_ring_commit(desc, _t(c["q"]), _t(c["qo"]), _t(c["k_chunk"]),
                                        _t(c["v_chunk"]), _t(c["k_ring"]), _t(c["v_ring"]),
                                        _t(c["ring_tab"]), _t(c["kv"]), 0.1, window, out,
                                        c["qo"], c["kv"], ws)
        assert e.value.status == 1
