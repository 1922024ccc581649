"""Small hand-built cases and textbook references for the oracle's pins.

A case starts from *logical* per-sequence K/V arrays and scatters them into a
paged pool through a random block table, so a dense reference computed from
the logical arrays never touches the paging the oracle must get right.
"""
from __future__ import annotations

import numpy as np
import scipy.special
import torch

BS = 16


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bits via torch's own rounding (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


class PagedCase:
    """Logical K/V per sequence, the pool they were scattered into, and q."""

    def __init__(self, rng, lens, hq, hkv, d, q_lens=None, num_blocks=None, fp8=False,
                 poison=False):
        self.lens = np.asarray(lens, dtype=np.int32)
        self.hq, self.hkv, self.d = hq, hkv, d
        self.q_lens = np.ones(len(lens), np.int32) if q_lens is None else np.asarray(q_lens,
                                                                                     np.int32)
        B = len(lens)
        nblk = (self.lens + BS - 1) // BS
        need = int(nblk.sum())
        nb = num_blocks or max(need + 3, 2 * need)
        self.num_blocks = nb
        perm = rng.permutation(nb)
        self.mbps = max(1, int(nblk.max()))
        self.tables = np.full((B, self.mbps), -1, np.int32)
        off = 0
        for s in range(B):
            self.tables[s, :nblk[s]] = perm[off:off + nblk[s]]
            off += nblk[s]
        self.fp8 = fp8
        # logical values
        self.K = [rng.standard_normal((n, hkv, d)).astype(np.float32) for n in self.lens]
        self.V = [rng.standard_normal((n, hkv, d)).astype(np.float32) for n in self.lens]
        fill = np.nan if poison else 0.0
        if fp8:
            amax_k = max(np.abs(k).max() for k in self.K)
            amax_v = max(np.abs(v).max() for v in self.V)
            self.k_scale = np.full(hkv, amax_k / 448.0, np.float32) * \
                (1 + 0.25 * np.arange(hkv, dtype=np.float32))
            self.v_scale = np.full(hkv, amax_v / 448.0, np.float32) * \
                (1 + 0.5 * np.arange(hkv, dtype=np.float32))
            self.Kc = [e4m3_codes(k / self.k_scale[None, :, None]) for k in self.K]
            self.Vc = [e4m3_codes(v / self.v_scale[None, :, None]) for v in self.V]
            self.k_cache = np.full((nb, hkv, BS, d), 0x7F if poison else 0, np.uint8)
            self.v_cache = np.full((nb, hkv, BS, d), 0x7F if poison else 0, np.uint8)
            srcK, srcV = self.Kc, self.Vc
        else:
            self.k_scale = self.v_scale = None
            self.Kb = [bf16_bits(k) for k in self.K]
            self.Vb = [bf16_bits(v) for v in self.V]
            self.k_cache = np.full((nb, hkv, BS, d), 0x7FC0 if poison else 0, np.uint16)
            self.v_cache = np.full((nb, hkv, BS, d), 0x7FC0 if poison else 0, np.uint16)
            srcK, srcV = self.Kb, self.Vb
        for s in range(B):
            for t in range(self.lens[s]):
                blk = self.tables[s, t // BS]
                self.k_cache[blk, :, t % BS, :] = srcK[s][t]
                self.v_cache[blk, :, t % BS, :] = srcV[s][t]
        del fill
        self.qo = np.zeros(B + 1, np.int32)
        self.qo[1:] = np.cumsum(self.q_lens)
        self.q = bf16_bits(rng.standard_normal((int(self.qo[-1]), hq, d)).astype(np.float32))

    # values exactly as the oracle must read them, in float64
    def k_f64(self, s):
        if self.fp8:
            return e4m3_to_f64(self.Kc[s]) * self.k_scale.astype(np.float64)[None, :, None]
        return bits_to_f64(self.Kb[s])

    def v_f64(self, s):
        if self.fp8:
            return e4m3_to_f64(self.Vc[s]) * self.v_scale.astype(np.float64)[None, :, None]
        return bits_to_f64(self.Vb[s])

    def oracle_kwargs(self):
        return dict(q=self.q, k_cache=self.k_cache, v_cache=self.v_cache,
                    block_tables=self.tables, qo_indptr=self.qo, kv_lens=self.lens,
                    num_q_heads=self.hq, num_kv_heads=self.hkv, kv_dtype=1 if self.fp8 else 0,
                    k_scale=self.k_scale, v_scale=self.v_scale)


def dense_reference(case: PagedCase, sm_scale, causal=True, window=-1):
    """Textbook softmax attention in float64 on the logical (contiguous) K/V,
    with an explicit boolean mask per query.  scipy's softmax / logsumexp."""
    T = int(case.qo[-1])
    out = np.zeros((T, case.hq, case.d))
    lse = np.full((T, case.hq), -np.inf)
    G = case.hq // case.hkv
    for s in range(len(case.lens)):
        K, V = case.k_f64(s), case.v_f64(s)
        n = int(case.lens[s])
        ql = int(case.q_lens[s])
        for j in range(ql):
            i = int(case.qo[s]) + j
            pos = n - ql + j
            t = np.arange(n)
            mask = np.ones(n, bool)
            if causal:
                mask &= t <= pos
            if window > 0:
                mask &= t > pos - window
            if not mask.any():
                continue
            qv = bits_to_f64(case.q[i])
            for h in range(case.hq):
                kh = h // G
                logits = sm_scale * (K[mask, kh, :] @ qv[h])
                p = scipy.special.softmax(logits)
                out[i, h] = p @ V[mask, kh, :]
                lse[i, h] = scipy.special.logsumexp(logits)
    return out, lse
