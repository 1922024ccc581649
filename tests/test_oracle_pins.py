"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against a library routine, a closed form, an
invariant the pages state, brute force on tiny inputs, or a value the pages
print (tests/golden/).  A plausible slip in the oracle -- a dropped term, a
wrong sign, a transposed index, a mask off by one -- fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from tests._cases import (BS, PagedCase, bf16_bits, bits_to_f64, dense_reference, e4m3_codes,
                          e4m3_to_f64)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def structured_f32_bits():
    """Every bf16 pattern (top 16 bits) times low-half patterns that sit on,
    just below and just above every rounding point at or above bit 16."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    return (hi[:, None] | lows[None, :]).reshape(-1)


# ----------------------------------------------------------- conversions --

def test_bf16_narrowing_matches_torch_rne():
    bits = structured_f32_bits()
    rnd = np.random.default_rng(1).integers(0, 2**32, size=1 << 20, dtype=np.uint64)
    bits = np.concatenate([bits, rnd.astype(np.uint32)])
    x = bits.view(np.float32)
    ours = oracle.bf16_from_f32(x)
    ref = bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    assert np.all(np.isnan(bits_to_f64(ours[nan])))


def test_bf16_widening_exact():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.f32_from_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(ours[nan]))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.f32_from_e4m3(codes)
    ref = e4m3_to_f64(codes).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7F and 0xFF only: E4M3FN has no infinities
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_encode_matches_torch_rne_in_range():
    bits = structured_f32_bits()
    rnd = np.random.default_rng(2).standard_normal(1 << 20).astype(np.float32) * 64
    x = np.concatenate([bits.view(np.float32), rnd])
    x = x[np.isfinite(x) & (np.abs(x) <= 464.0)]
    ours = oracle.e4m3_from_f32(x)
    ref = e4m3_codes(x)
    assert np.array_equal(ours, ref)


def test_e4m3_code_points_and_saturation():
    # OCP E4M3FN fixed points: exponent bias 7, max 448, min subnormal 2^-9.
    cases = {1.0: 0x38, 448.0: 0x7E, 2.0 ** -9: 0x01, -2.0: 0xC0, 0.5: 0x30, 2.0 ** -6: 0x08,
             7 * 2.0 ** -9: 0x07, 240.0: 0x77, 1000.0: 0x7E, -1e30: 0xFE, 0.0: 0x00,
             float("inf"): 0x7E, float("-inf"): 0xFE, 2.0 ** -10: 0x00, 1.0625: 0x38,
             1.1875: 0x3A}
    x = np.array(list(cases), np.float32)
    got = oracle.e4m3_from_f32(x)
    assert [int(v) for v in got] == list(cases.values())
    assert int(oracle.e4m3_from_f32(np.array([-0.0], np.float32))[0]) == 0x80
    assert int(oracle.e4m3_from_f32(np.array([np.nan], np.float32))[0]) & 0x7F == 0x7F


# ------------------------------------------------------------------ RoPE --

@pytest.mark.parametrize("theta,dim", [(1.0e6, 128), (1.0e4, 64), (5.0e5, 128)])
def test_rope_table_matches_numpy_double(theta, dim):
    P = 4096
    ours = oracle.rope_table(theta, dim, P)
    i = np.arange(dim // 2, dtype=np.float64)
    ang = np.arange(P, dtype=np.float64)[:, None] * np.power(float(np.float32(theta)),
                                                              -(2.0 * i) / dim)[None, :]
    ref_c = np.cos(ang).astype(np.float32)
    ref_s = np.sin(ang).astype(np.float32)
    # one rounding of a double: equal, or (on a near-tie) one fp32 ulp apart
    for got, ref in ((ours[..., 0], ref_c), (ours[..., 1], ref_s)):
        ulp = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
        assert ulp.max() <= 1
        assert (ulp == 0).mean() > 0.999
    assert np.all(ours[0, :, 0] == 1.0) and np.all(ours[0, :, 1] == 0.0)


def _append_one(x_bits, pos, table, hq=1, hkv=1):
    """Rotate one vector through the oracle's append (as a K row, no FP8)."""
    d = x_bits.shape[-1]
    kc = np.zeros((pos // BS + 1, hkv, BS, d), np.uint16)
    vc = np.zeros_like(kc)
    bt = np.arange(pos // BS + 1, dtype=np.int32)[None, :]
    oracle.append_rope(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS,
                       kv_dtype=0, k_cache=kc, v_cache=vc, block_tables=bt,
                       token_to_seq=[0], positions=[pos], k_new=x_bits.reshape(1, hkv, d),
                       v_new=x_bits.reshape(1, hkv, d), cos_sin=table)
    return kc[pos // BS, :, pos % BS, :].copy(), vc[pos // BS, :, pos % BS, :].copy()


def test_rope_position_zero_is_identity_and_v_is_untouched():
    rng = np.random.default_rng(3)
    table = oracle.rope_table(1e6, 128, 64)
    x = bf16_bits(rng.standard_normal((1, 128)).astype(np.float32))
    k, v = _append_one(x, 0, table)
    assert np.array_equal(k, x)
    k, v = _append_one(x, 37, table)
    assert np.array_equal(v, x)          # no RoPE on V
    assert not np.array_equal(k, x)


def test_rope_matches_complex_rotation():
    """Half-split RoPE is multiplication of z_i = x_i + i x_{i+D/2} by
    exp(i * angle_i): an independent statement of the same rotation."""
    rng = np.random.default_rng(4)
    d = 128
    table = oracle.rope_table(1e6, d, 3000)
    for pos in (1, 17, 255, 2999):
        x = bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
        k, _ = _append_one(x, pos, table)
        xf = bits_to_f64(x[0])
        z = xf[: d // 2] + 1j * xf[d // 2:]
        i = np.arange(d // 2)
        ang = pos * np.power(1e6, -(2.0 * i) / d)
        r = z * np.exp(1j * ang)
        ref = np.concatenate([r.real, r.imag])
        got = bits_to_f64(k[0])
        # bf16 output: within one bf16 ulp (2^-8 relative) of the exact value
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_rope_relative_position():
    """q_m . k_n depends only on m - n."""
    rng = np.random.default_rng(5)
    d = 64
    table = oracle.rope_table(1e4, d, 600)
    q = bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
    k = bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
    dots = []
    for shift in (0, 100, 333):
        qm, _ = _append_one(q, 40 + shift, table)
        kn, _ = _append_one(k, 7 + shift, table)
        dots.append(float(bits_to_f64(qm[0]) @ bits_to_f64(kn[0])))
    assert max(dots) - min(dots) <= 0.05 * max(1.0, abs(dots[0]))


def test_rope_composition():
    """Rotating by angle(a) then by angle(b) equals rotating by angle(a+b)."""
    rng = np.random.default_rng(6)
    d = 128
    table = oracle.rope_table(1e6, d, 400)
    x = bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
    ka, _ = _append_one(x, 150, table)
    kab, _ = _append_one(ka, 200, table)
    k_sum, _ = _append_one(x, 350, table)
    a, b = bits_to_f64(kab[0]), bits_to_f64(k_sum[0])
    assert np.all(np.abs(a - b) <= 2.0 ** -6 * np.maximum(np.abs(b), 0.25))


def test_append_places_q_k_v_and_rotates_q():
    rng = np.random.default_rng(7)
    hq, hkv, d, nb = 8, 2, 64, 12
    table = oracle.rope_table(1e4, d, 200)
    kc = np.zeros((nb, hkv, BS, d), np.uint16)
    vc = np.zeros_like(kc)
    bt = np.array([[5, 2, 9, -1], [0, 11, 3, 7]], np.int32)
    pos = np.array([33, 0, 63, 17], np.int32)
    seq = np.array([0, 1, 1, 0], np.int32)
    kn = bf16_bits(rng.standard_normal((4, hkv, d)).astype(np.float32))
    vn = bf16_bits(rng.standard_normal((4, hkv, d)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((4, hq, d)).astype(np.float32))
    qo = oracle.append_rope(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS,
                            kv_dtype=0, k_cache=kc, v_cache=vc, block_tables=bt, token_to_seq=seq,
                            positions=pos, k_new=kn, v_new=vn, q=q, cos_sin=table)
    written = np.zeros((nb, BS), bool)
    for i in range(4):
        blk = bt[seq[i], pos[i] // BS]
        written[blk, pos[i] % BS] = True
        assert np.array_equal(vc[blk, :, pos[i] % BS], vn[i])
        for h in range(hkv):
            k1, _ = _append_one(kn[i, h][None], int(pos[i]), table)
            assert np.array_equal(kc[blk, h, pos[i] % BS], k1[0])
        for h in range(hq):
            q1, _ = _append_one(q[i, h][None], int(pos[i]), table)
            assert np.array_equal(qo[i, h], q1[0])
    kt = kc.transpose(0, 2, 1, 3)  # [nb][bs][hkv][d]
    vt = vc.transpose(0, 2, 1, 3)
    assert not np.any(kt[~written]) and not np.any(vt[~written])


def test_append_then_gather_round_trip():
    rng = np.random.default_rng(8)
    hkv, d, nb = 3, 64, 40
    lens = np.array([5, 40, 16, 1], np.int32)
    case_tables = np.full((4, 3), -1, np.int32)
    perm = rng.permutation(nb)
    off = 0
    for s, n in enumerate((lens + BS - 1) // BS):
        case_tables[s, :n] = perm[off:off + n]
        off += n
    seq = np.concatenate([np.full(n, s, np.int32) for s, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    kn = bf16_bits(rng.standard_normal((len(seq), hkv, d)).astype(np.float32))
    vn = bf16_bits(rng.standard_normal((len(seq), hkv, d)).astype(np.float32))
    kc = np.zeros((nb, hkv, BS, d), np.uint16)
    vc = np.zeros_like(kc)
    oracle.append_rope(num_q_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=BS, kv_dtype=0,
                       k_cache=kc, v_cache=vc, block_tables=case_tables, token_to_seq=seq,
                       positions=pos, k_new=kn, v_new=vn)
    assert np.array_equal(oracle.gather_kv(kc, case_tables, lens, block_size=BS), kn)
    assert np.array_equal(oracle.gather_kv(vc, case_tables, lens, block_size=BS), vn)
    # gather against plain numpy indexing of the pool
    for s in range(4):
        t = np.arange(lens[s])
        ref = kc[case_tables[s, t // BS], :, t % BS, :]
        got = oracle.gather_kv(kc, case_tables[s:s + 1], lens[s:s + 1], block_size=BS)
        assert np.array_equal(got, ref)


def test_append_fp8_codes_match_torch_cast():
    rng = np.random.default_rng(9)
    hkv, d = 2, 64
    x = rng.standard_normal((3, hkv, d)).astype(np.float32) * 3
    x[0, 0, :4] = [2000.0, -2000.0, 1e-12, -1e-12]  # saturation and flush to zero
    kn = bf16_bits(x)
    vn = bf16_bits(x[::-1].copy())
    ks = np.array([0.01, 0.02], np.float32)
    vs = np.array([0.015, 0.005], np.float32)
    kc = np.zeros((4, hkv, BS, d), np.uint8)
    vc = np.zeros_like(kc)
    bt = np.array([[2, 0]], np.int32)
    oracle.append_rope(num_q_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=BS, kv_dtype=1,
                       k_cache=kc, v_cache=vc, block_tables=bt, token_to_seq=[0, 0, 0],
                       positions=[3, 16, 31], k_new=kn, v_new=vn, k_scale=ks, v_scale=vs)
    for i, p in enumerate((3, 16, 31)):
        blk = bt[0, p // BS]
        kf = bits_to_f64(kn[i]).astype(np.float32) / ks[:, None]
        vf = bits_to_f64(vn[i]).astype(np.float32) / vs[:, None]
        assert np.array_equal(kc[blk, :, p % BS], e4m3_codes(np.clip(kf, -448, 448)))
        assert np.array_equal(vc[blk, :, p % BS], e4m3_codes(np.clip(vf, -448, 448)))


# ------------------------------------------------------------- attention --

def _run(case, sm_scale, causal=True, window=-1, precision=32, nthreads=1):
    return oracle.paged_attention(**case.oracle_kwargs(), sm_scale=sm_scale, causal=causal,
                                  window=window, precision=precision, nthreads=nthreads)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (16, 2, 128), (4, 4, 32), (8, 1, 16)])
def test_decode_matches_dense_float64(hq, hkv, d):
    rng = np.random.default_rng(10 + hq + d)
    case = PagedCase(rng, [17, 64, 100, 255, 1, 16, 33], hq, hkv, d)
    sm = 1.0 / math.sqrt(d)
    out, lse = _run(case, sm)
    ref, ref_lse = dense_reference(case, sm)
    assert np.abs(out - ref).max() < 2e-6
    assert np.abs(lse - ref_lse).max() < 2e-5


def test_decode_matches_torch_sdpa():
    rng = np.random.default_rng(11)
    hq, hkv, d = 16, 4, 64
    case = PagedCase(rng, [40, 7, 129], hq, hkv, d)
    sm = 0.1
    out, _ = _run(case, sm)
    G = hq // hkv
    for s in range(3):
        K = torch.from_numpy(case.k_f64(s)).permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = torch.from_numpy(case.v_f64(s)).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qv = torch.from_numpy(bits_to_f64(case.q[s]))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qv, K, V, scale=sm)[:, 0, :]
        assert np.abs(out[s] - ref.numpy()).max() < 2e-6


def test_fp64_variant_bounds_fp32():
    rng = np.random.default_rng(12)
    case = PagedCase(rng, [300, 1000], 8, 2, 128)
    o32, l32 = _run(case, 1 / math.sqrt(128))
    o64, l64 = _run(case, 1 / math.sqrt(128), precision=64)
    ref, ref_lse = dense_reference(case, 1 / math.sqrt(128))
    assert np.abs(o64 - ref).max() < 1e-7
    assert np.abs(o32 - o64).max() < 5e-6


def test_block_placement_invariance_is_bit_exact():
    rng = np.random.default_rng(13)
    case = PagedCase(rng, [50, 130, 3], 8, 2, 64, num_blocks=40)
    o1, l1 = _run(case, 0.125)
    perm = np.random.default_rng(99).permutation(case.num_blocks)
    inv = np.argsort(perm)
    k2 = case.k_cache[perm]          # new block j holds old block perm[j]
    v2 = case.v_cache[perm]
    t2 = np.where(case.tables >= 0, inv[np.maximum(case.tables, 0)], -1).astype(np.int32)
    kw = case.oracle_kwargs()
    kw.update(k_cache=k2, v_cache=v2, block_tables=t2)
    o2, l2 = oracle.paged_attention(**kw, sm_scale=0.125)
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32))


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(14)
    case = PagedCase(rng, [70, 20, 300, 5], 8, 2, 64)
    o1, l1 = _run(case, 0.125, nthreads=1)
    o4, l4 = _run(case, 0.125, nthreads=5)
    assert np.array_equal(o1.view(np.uint32), o4.view(np.uint32))
    assert np.array_equal(l1.view(np.uint32), l4.view(np.uint32))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(15)
    case = PagedCase(rng, [37], 4, 1, 32)
    key = case.Kb[0][0].copy()
    for t in range(37):
        blk = case.tables[0, t // BS]
        case.k_cache[blk, :, t % BS, :] = key
    out, lse = _run(case, 0.3)
    mean_v = case.v_f64(0)[:, 0, :].mean(axis=0)
    assert np.abs(out[0] - mean_v[None, :]).max() < 1e-6
    # lse = l + ln(n) for equal logits l
    l = 0.3 * (bits_to_f64(case.q[0]) @ bits_to_f64(key[0]))
    assert np.abs(lse[0] - (l + math.log(37))).max() < 1e-5


def test_single_key_and_window_one_return_the_value_exactly():
    rng = np.random.default_rng(16)
    case = PagedCase(rng, [1, 9, 40], 4, 2, 64)
    out, lse = _run(case, 0.125, window=1)
    for s in range(3):
        v_last = case.v_f64(s)[-1]
        G = 2
        for h in range(4):
            assert np.array_equal(out[s, h].astype(np.float64), v_last[h // G])
    out1, _ = _run(case, 0.125)
    assert np.array_equal(out1[0].astype(np.float64), np.repeat(case.v_f64(0)[0], 2, axis=0))


def test_brute_force_tiny_all_masks():
    """Pure-Python softmax on ctx <= 4, D = 4 for every length, causal flag,
    window and query length."""
    rng = np.random.default_rng(17)
    for n, causal, window, ql in itertools.product(range(1, 5), (True, False), (-1, 1, 2, 3),
                                                   range(1, 3)):
        if ql > n:
            continue
        case = PagedCase(rng, [n], 2, 1, 4, q_lens=[ql])
        out, lse = _run(case, 0.7, causal=causal, window=window)
        K, V = case.k_f64(0)[:, 0, :].tolist(), case.v_f64(0)[:, 0, :].tolist()
        for j in range(ql):
            pos = n - ql + j
            vis = [t for t in range(n) if (not causal or t <= pos) and
                   (window <= 0 or t > pos - window)]
            for h in range(2):
                qv = bits_to_f64(case.q[j, h]).tolist()
                logit = [0.7 * sum(a * b for a, b in zip(qv, K[t])) for t in vis]
                if not vis:
                    assert np.all(out[j, h] == 0) and lse[j, h] == -np.inf
                    continue
                mx = max(logit)
                w = [math.exp(x - mx) for x in logit]
                tot = sum(w)
                ref = [sum(w[i] * V[t][c] for i, t in enumerate(vis)) / tot for c in range(4)]
                assert max(abs(a - b) for a, b in zip(out[j, h], ref)) < 1e-6
                assert abs(lse[j, h] - (mx + math.log(tot))) < 1e-5


def test_prefill_causal_matches_sdpa_is_causal():
    rng = np.random.default_rng(18)
    hq, hkv, d, n = 8, 2, 32, 45
    case = PagedCase(rng, [n], hq, hkv, d, q_lens=[n])
    out, _ = _run(case, 0.2)
    G = hq // hkv
    K = torch.from_numpy(case.k_f64(0)).permute(1, 0, 2).repeat_interleave(G, dim=0)
    V = torch.from_numpy(case.v_f64(0)).permute(1, 0, 2).repeat_interleave(G, dim=0)
    Q = torch.from_numpy(bits_to_f64(case.q)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=0.2)
    assert np.abs(out - ref.permute(1, 0, 2).numpy()).max() < 2e-6


@pytest.mark.parametrize("causal,window", [(True, -1), (True, 128), (True, 7), (False, 7),
                                           (False, 128)])
def test_ragged_prefill_over_prefix_matches_dense(causal, window):
    """Without causality a windowed query sees [p - W + 1, kv_len): more than
    W keys, the case that sizes the oracle's per-worker logit buffer."""
    rng = np.random.default_rng(19)
    case = PagedCase(rng, [200, 37, 64, 300], 8, 2, 64, q_lens=[50, 37, 1, 16])
    out, lse = _run(case, 0.125, causal=causal, window=window)
    ref, ref_lse = dense_reference(case, 0.125, causal=causal, window=window)
    assert np.abs(out - ref).max() < 2e-6
    assert np.abs(lse - ref_lse).max() < 2e-5


def test_decode_window_matches_dense():
    rng = np.random.default_rng(20)
    case = PagedCase(rng, [1024, 130, 128, 129, 5], 16, 2, 64)
    out, _ = _run(case, 0.125, window=128)
    ref, _ = dense_reference(case, 0.125, window=128)
    assert np.abs(out - ref).max() < 2e-6


def test_fp8_decode_matches_dense_on_dequantised_values():
    rng = np.random.default_rng(21)
    case = PagedCase(rng, [17, 300, 1000], 16, 2, 64, fp8=True)
    for window in (-1, 128):
        out, lse = _run(case, 0.125, window=window)
        ref, ref_lse = dense_reference(case, 0.125, window=window)
        assert np.abs(out - ref).max() < 2e-6
        assert np.abs(lse - ref_lse).max() < 2e-5


def test_unused_slots_do_not_matter():
    rng = np.random.default_rng(22)
    a = PagedCase(rng, [19, 70], 8, 2, 64, poison=True)
    out, _ = _run(a, 0.125)
    assert np.all(np.isfinite(out))
    ref, _ = dense_reference(a, 0.125)
    assert np.abs(out - ref).max() < 2e-6


def test_chunked_prefill_equals_one_shot_bit_exact():
    """Chunked prefill == one-shot prefill, difference 0.0 (the value the
    infer-lab page prints in its verified-invariants table)."""
    with open(os.path.join(GOLDEN, "chunked_vs_oneshot.json")) as f:
        gold = json.load(f)
    rng = np.random.default_rng(23)
    n = 300
    case = PagedCase(rng, [n], 8, 2, 64, q_lens=[n])
    full, full_lse = _run(case, 0.125)
    pieces, pieces_lse = [], []
    for a, b in ((0, 64), (64, 65), (65, 200), (200, 300)):
        kw = case.oracle_kwargs()
        kw.update(q=case.q[a:b], qo_indptr=np.array([0, b - a], np.int32),
                  kv_lens=np.array([b], np.int32))
        o, l = oracle.paged_attention(**kw, sm_scale=0.125)
        pieces.append(o)
        pieces_lse.append(l)
    diff = float(np.abs(np.concatenate(pieces) - full).max())
    assert diff == gold["max_abs_difference"]
    assert np.array_equal(np.concatenate(pieces_lse).view(np.uint32), full_lse.view(np.uint32))


# ----------------------------------------------------------------- merge --

def _split_case(rng, n, cuts, hq=8, hkv=2, d=64):
    """One sequence of n keys and the same keys cut into parts, each part a
    sequence of its own with the same query (q_len 1, non-causal)."""
    whole = PagedCase(rng, [n], hq, hkv, d)
    parts = []
    bounds = [0] + list(cuts) + [n]
    for a, b in zip(bounds[:-1], bounds[1:]):
        p = PagedCase(np.random.default_rng(0), [b - a], hq, hkv, d)
        for t in range(b - a):
            blk = p.tables[0, t // BS]
            p.k_cache[blk, :, t % BS] = whole.Kb[0][a + t]
            p.v_cache[blk, :, t % BS] = whole.Vb[0][a + t]
        p.q = whole.q.copy()
        parts.append(p)
    return whole, parts


def test_merge_of_split_equals_whole():
    rng = np.random.default_rng(24)
    whole, parts = _split_case(rng, 333, (100, 101, 250))
    o_full, l_full = _run(whole, 0.125, causal=False)
    os_, ls_ = zip(*[_run(p, 0.125, causal=False) for p in parts])
    o, l = oracle.merge_states(np.stack(os_), np.stack(ls_))
    assert np.abs(o - o_full).max() < 2e-6
    assert np.abs(l - l_full).max() < 2e-5


def test_merge_empty_part_is_identity_and_order_does_not_matter():
    rng = np.random.default_rng(25)
    whole, parts = _split_case(rng, 90, (30, 60))
    os_, ls_ = zip(*[_run(p, 0.125, causal=False) for p in parts])
    o_parts, l_parts = np.stack(os_), np.stack(ls_)
    empty_o = np.full_like(o_parts[:1], np.nan)  # an empty part's o is never read
    empty_l = np.full_like(l_parts[:1], -np.inf)
    o1, l1 = oracle.merge_states(o_parts[:1], l_parts[:1])
    o2, l2 = oracle.merge_states(np.concatenate([o_parts[:1], empty_o]),
                                 np.concatenate([l_parts[:1], empty_l]))
    assert np.array_equal(o1, o_parts[0]) and np.array_equal(o1, o2)
    assert np.array_equal(l1, l2) and np.array_equal(l1, l_parts[0])
    oa, la = oracle.merge_states(o_parts, l_parts)
    ob, lb = oracle.merge_states(o_parts[::-1], l_parts[::-1])
    assert np.abs(oa - ob).max() < 1e-6
    # associativity: merge(merge(a, b), c) == merge(a, b, c)
    oab, lab = oracle.merge_states(o_parts[:2], l_parts[:2])
    oc, lc = oracle.merge_states(np.stack([oab, o_parts[2]]), np.stack([lab, l_parts[2]]))
    assert np.abs(oc - oa).max() < 1e-6 and np.abs(lc - la).max() < 1e-5
    # all parts empty
    oz, lz = oracle.merge_states(np.zeros_like(o_parts), np.full_like(l_parts, -np.inf))
    assert np.all(oz == 0) and np.all(lz == -np.inf)


def test_lse_matches_scipy_logsumexp():
    rng = np.random.default_rng(26)
    case = PagedCase(rng, [500], 4, 1, 64)
    _, lse = _run(case, 0.125)
    K = case.k_f64(0)[:, 0, :]
    for h in range(4):
        logits = 0.125 * K @ bits_to_f64(case.q[0, h])
        assert abs(lse[0, h] - scipy.special.logsumexp(logits)) < 2e-5


def test_copy_blocks_matches_numpy_assignment():
    rng = np.random.default_rng(27)
    pool = rng.integers(0, 65535, size=(20, 2, BS, 16), dtype=np.uint16)
    ref = pool.copy()
    src = np.array([3, 3, 7, 19], np.int32)
    dst = np.array([0, 11, 12, 5], np.int32)
    ref[dst] = ref[src]
    oracle.copy_blocks(pool, src, dst)
    assert np.array_equal(pool, ref)


# ---------------------------------------------- sinks and the ring cache --

def test_sinks_equal_softmax_with_an_extra_zero_value_entry():
    """A sink logit s joins the softmax with a zero value vector: scipy's
    softmax / logsumexp over [logits, s] in float64, dropping the sink's row."""
    rng = np.random.default_rng(30)
    hq, hkv, d = 8, 2, 64
    case = PagedCase(rng, [1, 40, 130], hq, hkv, d)
    sinks = np.array([-3.0, 0.0, 1.5, 4.0, -np.inf, 2.0, 8.0, -1.0], np.float32)
    sm = 0.125
    out, lse = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=sm, sinks=sinks)
    G = hq // hkv
    for s in range(3):
        K, V = case.k_f64(s), case.v_f64(s)
        qv = bits_to_f64(case.q[s])
        for h in range(hq):
            logits = np.append(sm * (K[:, h // G, :] @ qv[h]), float(sinks[h]))
            p = scipy.special.softmax(logits)
            ref = p[:-1] @ V[:, h // G, :]
            assert np.abs(out[s, h] - ref).max() < 2e-6
            assert abs(lse[s, h] - scipy.special.logsumexp(logits)) < 2e-5


def test_sink_of_minus_infinity_changes_no_bit_and_a_large_sink_takes_the_mass():
    rng = np.random.default_rng(31)
    case = PagedCase(rng, [50, 7], 4, 2, 32)
    o0, l0 = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=0.2)
    o1, l1 = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=0.2,
                                    sinks=np.full(4, -np.inf, np.float32))
    assert np.array_equal(o0.view(np.uint32), o1.view(np.uint32))
    assert np.array_equal(l0.view(np.uint32), l1.view(np.uint32))
    o2, l2 = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=0.2,
                                    sinks=np.full(4, 60.0, np.float32))
    assert np.abs(o2).max() < 1e-9  # every key weighs about e^-60 against the sink
    assert np.abs(l2 - 60.0).max() < 1e-5


def _ring_from_linear(case, ring):
    """A ring pool of `ring` blocks per sequence holding, in entry b % ring,
    the last logical block b that maps there (numpy copies)."""
    B = len(case.lens)
    nb = B * ring
    k = np.zeros((nb,) + case.k_cache.shape[1:], case.k_cache.dtype)
    v = np.zeros_like(k)
    tabs = np.full((B, ring), -1, np.int32)
    for s in range(B):
        tabs[s] = np.arange(ring) + s * ring
        for b in range((int(case.lens[s]) + BS - 1) // BS):
            k[tabs[s, b % ring]] = case.k_cache[case.tables[s, b]]
            v[tabs[s, b % ring]] = case.v_cache[case.tables[s, b]]
    return k, v, tabs


@pytest.mark.parametrize("window,ring", [(128, 9), (40, 4), (16, 2)])
def test_ring_cache_equals_the_linear_cache_over_the_window(window, ring):
    rng = np.random.default_rng(32 + window)
    case = PagedCase(rng, [1, 15, 16, 17, 130, 700, 1031], 8, 2, 64)
    o_lin, l_lin = oracle.paged_attention(**case.oracle_kwargs(), sm_scale=0.125, window=window)
    k, v, tabs = _ring_from_linear(case, ring)
    kw = case.oracle_kwargs()
    kw.update(k_cache=k, v_cache=v, block_tables=tabs)
    o_ring, l_ring = oracle.paged_attention(**kw, sm_scale=0.125, window=window, ring_blocks=ring)
    assert np.array_equal(o_lin.view(np.uint32), o_ring.view(np.uint32))
    assert np.array_equal(l_lin.view(np.uint32), l_ring.view(np.uint32))
    ref, _ = dense_reference(case, 0.125, window=window)
    assert np.abs(o_ring - ref).max() < 2e-6
    # a ring too small for the window is refused
    with pytest.raises(Exception):
        oracle.paged_attention(**kw, sm_scale=0.125, window=window + BS, ring_blocks=ring)


def test_ring_append_writes_entry_block_mod_ring():
    rng = np.random.default_rng(33)
    hkv, d, ring, n = 2, 32, 3, 100
    kc = np.zeros((ring, hkv, BS, d), np.uint16)
    vc = np.zeros_like(kc)
    tab = np.array([[2, 0, 1]], np.int32)
    kn = bf16_bits(rng.standard_normal((n, hkv, d)))
    vn = bf16_bits(rng.standard_normal((n, hkv, d)))
    for p in range(n):
        oracle.append_rope(num_q_heads=hkv, num_kv_heads=hkv, head_dim=d, block_size=BS,
                           kv_dtype=oracle.KV_BF16, k_cache=kc, v_cache=vc, block_tables=tab,
                           token_to_seq=[0], positions=[p], k_new=kn[p:p + 1], v_new=vn[p:p + 1],
                           ring_blocks=ring)
    for p in range(n):
        b = p // BS
        if b >= (n - 1) // BS - ring + 1:  # not yet overwritten by a later block
            assert np.array_equal(kc[tab[0, b % ring], :, p % BS], kn[p])
            assert np.array_equal(vc[tab[0, b % ring], :, p % BS], vn[p])
