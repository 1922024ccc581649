"""GPU parity of cascade (shared-prefix) decode: groups of sequences share a
cached prefix, each has its own suffix; the result must equal attention over
the concatenated keys (infer-lab's invariant "prefix-cached == uncached"),
checked against the oracle element by element and against the plain decode
over the concatenated table -- over bf16 and e4m3 pools, with full attention
and with sliding windows that reach none, part or all of the prefix."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import DEV, NTHREADS, assert_close, assert_lse_close, gpu_decode, pool_np, u16

pytestmark = pytest.mark.gpu

BS = 16


def _case(hq, hkv, d, group_sizes, prefix_lens, suffix_hi, seed, fp8=False):
    """A pool with per-group prefix blocks and per-sequence suffix blocks (test
    plumbing: index bookkeeping only)."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    ng = len(group_sizes)
    n = int(sum(group_sizes))
    suffix_lens = rng.integers(1, suffix_hi + 1, size=n).astype(np.int32)
    pblocks = [(p + BS - 1) // BS for p in prefix_lens]
    sblocks = [(s + BS - 1) // BS for s in suffix_lens]
    mbps = max(max(pblocks + [1]), max(sblocks))
    nb = int(sum(pblocks) + sum(sblocks)) + 7
    ids = rng.permutation(nb).astype(np.int32)
    if fp8:
        k, ks = wl.fill_e4m3((nb, hkv, BS, d), gen, "cpu")
        v, vs = wl.fill_e4m3((nb, hkv, BS, d), gen, "cpu")
    else:
        k, ks = wl.fill_bf16((nb, hkv, BS, d), gen, "cpu"), None
        v, vs = wl.fill_bf16((nb, hkv, BS, d), gen, "cpu"), None
    ptab = np.full((ng, mbps), -1, np.int32)
    stab = np.full((n, mbps), -1, np.int32)
    off = 0
    for g in range(ng):
        ptab[g, :pblocks[g]] = ids[off:off + pblocks[g]]
        off += pblocks[g]
    for s in range(n):
        stab[s, :sblocks[s]] = ids[off:off + sblocks[s]]
        off += sblocks[s]
    q = wl.fill_bf16((n, hq, d), gen, "cpu")
    gptr = np.zeros(ng + 1, np.int32)
    gptr[1:] = np.cumsum(group_sizes)
    return dict(k=k, v=v, ks=ks, vs=vs, q=q, ptab=ptab, stab=stab,
                plen=np.asarray(prefix_lens, np.int32), slen=suffix_lens, gptr=gptr, mbps=mbps,
                fp8=fp8)


def _concatenated(c, hkv, d):
    """Each sequence's prefix keys followed by its suffix keys, in a fresh pool
    of consecutive blocks (numpy gathers of the bf16 bits)."""
    kb = pool_np(c["k"])
    vb = pool_np(c["v"])
    n = len(c["slen"])
    seq_k, seq_v, lens = [], [], []
    for g in range(len(c["plen"])):
        for s in range(c["gptr"][g], c["gptr"][g + 1]):
            toks_k, toks_v = [], []
            for tab, ln in ((c["ptab"][g], c["plen"][g]), (c["stab"][s], c["slen"][s])):
                for t in range(ln):
                    toks_k.append(kb[tab[t // BS], :, t % BS, :])
                    toks_v.append(vb[tab[t // BS], :, t % BS, :])
            seq_k.append(np.stack(toks_k, 1))
            seq_v.append(np.stack(toks_v, 1))
            lens.append(len(toks_k))
    lens = np.asarray(lens, np.int32)
    nblk = (lens + BS - 1) // BS
    mb = int(nblk.max())
    pool_k = np.zeros((int(nblk.sum()), hkv, BS, d), kb.dtype)
    pool_v = np.zeros_like(pool_k)
    tabs = np.full((n, mb), -1, np.int32)
    off = 0
    for s in range(n):
        for j in range(nblk[s]):
            a, b = j * BS, min(lens[s], (j + 1) * BS)
            pool_k[off, :, :b - a] = seq_k[s][:, a:b]
            pool_v[off, :, :b - a] = seq_v[s][:, a:b]
            tabs[s, j] = off
            off += 1
    return pool_k, pool_v, tabs, lens


@pytest.mark.parametrize("hq,hkv,d,fp8,window,big", [
    (32, 8, 128, False, -1, False), (16, 2, 128, False, -1, False), (8, 2, 64, False, -1, False),
    (32, 8, 128, True, -1, False), (64, 8, 64, True, -1, False), (32, 8, 128, True, -1, True),
    (64, 8, 64, True, -1, True),
    (32, 8, 128, False, 128, False), (16, 2, 128, False, 40, False), (64, 8, 64, True, 128, False),
    (8, 2, 64, True, 2000, False)])
def test_cascade_equals_attention_over_the_concatenated_keys(hq, hkv, d, fp8, window, big):
    # big: groups of more than 64 query rows, so the prefix pass runs the tcgen05 kernel
    groups = [20, 3, 33, 2, 6] if big else [1, 3, 8, 2, 6]
    prefixes = [0, 160, 515, 1000, 33]  # none, aligned, unaligned, long, short
    c = _case(hq, hkv, d, groups, prefixes, 300, seed=41, fp8=fp8)
    n = int(sum(groups))
    desc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=c["k"].shape[0],
                         max_blocks_per_seq=c["mbps"], kv_dtype=1 if fp8 else 0)
    sm_scale = 1.0 / np.sqrt(d)
    max_suffix = int(c["slen"].max())
    ws = torch.zeros(max(pkv.pkv_cascade_workspace_size(desc, len(groups), n, max(prefixes),
                                                        max_suffix, window), 256),
                     dtype=torch.uint8, device=DEV)
    ks = None if c["ks"] is None else c["ks"].to(DEV)
    vs = None if c["vs"] is None else c["vs"].to(DEV)
    out = torch.full((n, hq, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n, hq), float("nan"), device=DEV)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    kd, vd = c["k"].to(DEV), c["v"].to(DEV)
    for _ in range(2):  # twice: the workspace is reused
        pkv.pkv_cascade_decode(desc, c["q"].to(DEV), kd, vd, t(c["gptr"]), c["gptr"], t(c["ptab"]),
                               t(c["plen"]), c["plen"], t(c["stab"]), t(c["slen"]), max_suffix,
                               sm_scale, out, lse, ws, window=window, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        pk, pv, tabs, lens = _concatenated(c, hkv, d)
        ref, ref_lse = oracle.paged_attention(
            q=u16(c["q"]), k_cache=pk, v_cache=pv, block_tables=tabs, qo_indptr=np.arange(n + 1),
            kv_lens=lens, num_q_heads=hq, num_kv_heads=hkv, sm_scale=sm_scale, causal=True,
            window=window, kv_dtype=1 if fp8 else 0,
            k_scale=None if ks is None else c["ks"].numpy(),
            v_scale=None if vs is None else c["vs"].numpy(), nthreads=NTHREADS)
        what = "cascade %d/%d/%d %s window %d" % (hq, hkv, d, "e4m3" if fp8 else "bf16", window)
        # a window of 40 over suffixes of 1..300 keys: some outputs average a handful of keys
        assert_close(out, ref, what, literal=window < 0 or window >= 128)
        assert_lse_close(lse, ref_lse, what)
    assert pkv.pkv_device_errors() == 0
    # the plain decode over the concatenated table agrees within the same bound
    cdesc = pkv.make_desc(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=pk.shape[0],
                          max_blocks_per_seq=tabs.shape[1], kv_dtype=1 if fp8 else 0)
    pool = (lambda a: t(a)) if fp8 else (lambda a: t(a).view(torch.bfloat16))
    dd = dict(q=c["q"].to(DEV), k_cache=pool(pk), v_cache=pool(pv),
              k_scale=ks, v_scale=vs, block_tables=t(tabs), context_lens=t(lens))
    plain, _, _ = gpu_decode(cdesc, dd, int(lens.max()), sm_scale, window=window)
    err = (plain.float() - out.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 1e-3


def test_cascade_rejects_bad_groups():
    desc = pkv.make_desc(num_q_heads=8, num_kv_heads=2, head_dim=64, num_blocks=10,
                         max_blocks_per_seq=4)
    q = torch.zeros((3, 8, 64), dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(16, dtype=torch.int32, device=DEV)
    kv = torch.zeros((10, 2, 16, 64), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkv.PkvError):  # group pointers do not end at num_seqs
        pkv.pkv_cascade_decode(desc, q, kv, kv, z, np.array([0, 2], np.int32), z, z,
                               np.array([0], np.int32), z, z, 4, 0.1, out, None, ws)
    fdesc = pkv.make_desc(num_q_heads=8, num_kv_heads=2, head_dim=64, num_blocks=10,
                          max_blocks_per_seq=4, kv_dtype=1)
    with pytest.raises(pkv.PkvError):  # e4m3 pools without scales
        pkv.pkv_cascade_decode(fdesc, q, z, z, z, np.array([0, 3], np.int32), z, z,
                               np.array([10], np.int32), z, z, 4, 0.1, out, None, ws)
    with pytest.raises(pkv.PkvError):  # prefix longer than a table row
        pkv.pkv_cascade_decode(desc, q, kv, kv, z, np.array([0, 3], np.int32), z, z,
                               np.array([65], np.int32), z, z, 4, 0.1, out, None, ws)
