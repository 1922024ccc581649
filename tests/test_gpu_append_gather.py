"""GPU parity, bit-exact: fused KV append + RoPE (bf16 and e4m3), the device
conversions it relies on, and the block-table gather."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_21_gb300 as pkv
from paged_kv_attention_21_gb300 import workloads as wl
from tests._gpu import DEV, desc_for, on_device, pool_np, u16, u8

pytestmark = pytest.mark.gpu


def _append_case(spec, fp8, rope=True, tokens_per_seq=1):
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    B = spec.batch
    seq = np.repeat(np.arange(B, dtype=np.int32), tokens_per_seq)
    pos = np.concatenate([b.lens_host[s] - tokens_per_seq + np.arange(tokens_per_seq)
                          for s in range(B)]).astype(np.int32)
    g = torch.Generator().manual_seed(77)
    T = len(seq)
    kn = wl.fill_bf16((T, spec.num_kv_heads, spec.head_dim), g, "cpu")
    vn = wl.fill_bf16((T, spec.num_kv_heads, spec.head_dim), g, "cpu") * 3
    qn = wl.fill_bf16((T, spec.num_q_heads, spec.head_dim), g, "cpu")
    max_pos = int(b.lens_host.max()) + 1
    table = oracle.rope_table(spec.rope_theta, spec.head_dim, max_pos) if rope else None
    return b, d, seq, pos, kn, vn, qn, table


@pytest.mark.parametrize("cfg,fp8,tps", [(1, False, 1), (3, False, 1), (1, False, 5), (5, True, 1),
                                         (5, True, 3)])
def test_append_rope_bit_exact(cfg, fp8, tps):
    spec = wl.CONFIGS[cfg]
    if cfg == 5:
        spec = wl.scaled(spec, batch=16, ctx_hi=2048)
    elif cfg == 3:
        pass  # full size: 256 tokens
    b, d, seq, pos, kn, vn, qn, table = _append_case(spec, fp8, tokens_per_seq=tps)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    qd = qn.to(DEV)
    pkv.pkv_append_rope(desc, d["k_cache"], d["v_cache"], d["block_tables"],
                        torch.from_numpy(seq).to(DEV), torch.from_numpy(pos).to(DEV), kn.to(DEV),
                        vn.to(DEV), q=qd, cos_sin=torch.from_numpy(table).to(DEV),
                        k_scale=d["k_scale"], v_scale=d["v_scale"])
    torch.cuda.synchronize()
    kh, vh = pool_np(b.k_cache).copy(), pool_np(b.v_cache).copy()
    ks = None if b.k_scale is None else b.k_scale.numpy()
    vs = None if b.v_scale is None else b.v_scale.numpy()
    qh = oracle.append_rope(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                            head_dim=spec.head_dim, block_size=16, kv_dtype=1 if fp8 else 0,
                            k_cache=kh, v_cache=vh, block_tables=b.tables_host, token_to_seq=seq,
                            positions=pos, k_new=u16(kn), v_new=u16(vn), q=u16(qn),
                            cos_sin=table, k_scale=ks, v_scale=vs)
    assert np.array_equal(pool_np(d["k_cache"]), kh)
    assert np.array_equal(pool_np(d["v_cache"]), vh)
    assert np.array_equal(u16(qd), qh)
    assert pkv.pkv_device_errors() == 0


def test_append_without_rope_is_a_copy():
    spec = wl.TINY
    b, d, seq, pos, kn, vn, qn, _ = _append_case(spec, False, rope=False)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    qd = qn.to(DEV)
    pkv.pkv_append_rope(desc, d["k_cache"], d["v_cache"], d["block_tables"],
                        torch.from_numpy(seq).to(DEV), torch.from_numpy(pos).to(DEV), kn.to(DEV),
                        vn.to(DEV), q=qd)
    lens = torch.from_numpy(b.lens_host).to(DEV)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(b.lens_host)]).astype(np.int32)).to(DEV)
    total = int(b.lens_host.sum())
    kg = torch.empty((total, spec.num_kv_heads, spec.head_dim), dtype=torch.bfloat16, device=DEV)
    pkv.pkv_gather_kv(desc, d["k_cache"], d["block_tables"], lens, cu, total, kg)
    torch.cuda.synchronize()
    last = np.cumsum(b.lens_host) - 1
    assert np.array_equal(u16(kg)[last], u16(kn))
    assert np.array_equal(u16(qd), u16(qn))  # no table: q untouched


def _structured_f32():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    rnd = np.random.default_rng(3).integers(0, 2 ** 32, size=1 << 18, dtype=np.uint64)
    x = np.concatenate([bits, rnd.astype(np.uint32)]).view(np.float32)
    return x[~np.isnan(x)]


@pytest.mark.parametrize("fp8", [False, True])
def test_device_rounding_matches_oracle_on_every_rounding_point(fp8):
    """The append kernel with k = 1 and a cos/sin table whose cos entries are
    arbitrary floats and sin entries 0 writes RNE(c) (bf16) or
    RNE-satfinite(c / 1) (e4m3): the device conversions, checked against the
    oracle's encoders on every bf16 pattern times the low-bit patterns that
    sit on and beside each rounding point."""
    x = _structured_f32()
    D = 64
    half = D // 2
    npos = (len(x) + half - 1) // half
    xs = np.zeros(npos * half, np.float32)
    xs[:len(x)] = x
    table = np.zeros((npos, half, 2), np.float32)
    table[:, :, 0] = xs.reshape(npos, half)
    nblk = (npos + 15) // 16
    kc = torch.zeros((nblk, 1, 16, D), dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    desc = pkv.make_desc(num_q_heads=1, num_kv_heads=1, head_dim=D, num_blocks=nblk,
                         max_blocks_per_seq=nblk, kv_dtype=1 if fp8 else 0)
    bt = torch.arange(nblk, dtype=torch.int32, device=DEV)[None, :]
    ones = torch.ones((npos, 1, D), dtype=torch.bfloat16, device=DEV)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    pkv.pkv_append_rope(desc, kc, vc, bt, torch.zeros(npos, dtype=torch.int32, device=DEV),
                        torch.arange(npos, dtype=torch.int32, device=DEV), ones, ones,
                        cos_sin=torch.from_numpy(table).to(DEV), k_scale=one, v_scale=one)
    torch.cuda.synchronize()
    k = (u8(kc) if fp8 else u16(kc)).reshape(nblk * 16, D)[:npos]
    lo = k[:, :half].reshape(-1)[:len(x)]   # a*c - b*s = c
    hi_ = k[:, half:].reshape(-1)[:len(x)]  # b*c + a*s = c
    ref = oracle.e4m3_from_f32(x) if fp8 else oracle.bf16_from_f32(x)
    assert np.array_equal(lo, ref)
    keep = ~((x == 0) & np.signbit(x))  # b*c + a*s turns c = -0 into +0
    assert np.array_equal(hi_[keep], ref[keep])


@pytest.mark.parametrize("cfg", [1, 2, 5])
def test_gather_bit_exact(cfg):
    spec = wl.CONFIGS[cfg]
    if cfg != 1:
        spec = wl.scaled(spec, batch=12, ctx_hi=min(spec.ctx_hi, 3000))
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    lens = d["context_lens"]
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(b.lens_host)]).astype(np.int32)).to(DEV)
    total = int(b.lens_host.sum())
    for name in ("k_cache", "v_cache"):
        out = torch.empty((total, spec.num_kv_heads, spec.head_dim), dtype=d[name].dtype,
                          device=DEV)
        pkv.pkv_gather_kv(desc, d[name], d["block_tables"], lens, cu, total, out)
        torch.cuda.synchronize()
        ref = oracle.gather_kv(pool_np(getattr(b, name)), b.tables_host, b.lens_host,
                               block_size=16)
        assert np.array_equal(pool_np(out), ref)


def test_bad_block_id_is_flagged_not_faulted():
    spec = wl.TINY
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    pkv.pkv_device_errors(reset=True)
    bt = d["block_tables"].clone()
    bt[1, 0] = 10 ** 6      # outside the pool
    seq = torch.tensor([1], dtype=torch.int32, device=DEV)
    pos = torch.tensor([3], dtype=torch.int32, device=DEV)
    kn = torch.zeros((1, spec.num_kv_heads, spec.head_dim), dtype=torch.bfloat16, device=DEV)
    before = pool_np(d["k_cache"]).copy()
    pkv.pkv_append_rope(desc, d["k_cache"], d["v_cache"], bt, seq, pos, kn, kn)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_BLOCK_ID
    assert np.array_equal(pool_np(d["k_cache"]), before)  # the write was skipped
    # a position beyond the table
    pos2 = torch.tensor([10 ** 5], dtype=torch.int32, device=DEV)
    pkv.pkv_append_rope(desc, d["k_cache"], d["v_cache"], d["block_tables"], seq, pos2, kn, kn)
    assert pkv.pkv_device_errors(reset=True) & pkv.DEVERR_POSITION
    assert pkv.pkv_device_errors() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_copy_blocks_bit_exact(fp8):
    spec = wl.scaled(wl.FP8_DECODE if fp8 else wl.QWEN3_4B, batch=8, ctx_hi=500)
    b = wl.make_decode_batch(spec, "cpu")
    d = on_device(b)
    desc = desc_for(spec, b.k_cache, b.tables_host)
    nb = b.k_cache.shape[0]
    rng = np.random.default_rng(5)
    perm = rng.permutation(nb)
    src, dst = perm[:40].astype(np.int32), perm[40:80].astype(np.int32)
    src[1] = src[0]  # one source shared by two copies
    pkv.pkv_copy_blocks(desc, d["k_cache"], d["v_cache"], torch.from_numpy(src).to(DEV),
                        torch.from_numpy(dst).to(DEV))
    torch.cuda.synchronize()
    kh, vh = pool_np(b.k_cache).copy(), pool_np(b.v_cache).copy()
    oracle.copy_blocks(kh, src, dst)
    oracle.copy_blocks(vh, src, dst)
    assert np.array_equal(pool_np(d["k_cache"]), kh)
    assert np.array_equal(pool_np(d["v_cache"]), vh)
    assert pkv.pkv_device_errors() == 0
