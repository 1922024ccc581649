/*
 * pkv_oracle.c -- plain, slow, obviously-correct CPU oracle for attention over
 * a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load or call this
 * file: only tests/, __graft_entry__.smoke() and the cpu_baseline leg of
 * bench.py (and its "--impl reference" arm) use it.  It shares no code, header,
 * table or constant generator with the CUDA library; neither includes the
 * other.
 *
 * What it computes, and where the pages state it:
 *   - paged KV storage addressed through per-sequence block tables
 *     (infer-lab, "Technique" table: PagedAttention -- block allocator, block
 *     tables, refcounting, copy-on-write; llm-infer, "What It Does": paged KV
 *     cache with block tables);
 *   - the KV write of each new token fused with RoPE (llm-infer, "What It
 *     Does": graphs capture KV writes; fused RMSNorm and RoPE; infer-lab
 *     source layout: Llama-style decoder with RMSNorm, RoPE, GQA);
 *   - FP8 e4m3 KV cache with frozen per-head scales (InferX, "The kernels
 *     underneath": M8's FP8 KV cache, scales frozen from warmup);
 *   - softmax attention over the gathered keys, the definition that the
 *     tiled/online forms must equal (infer-lab, invariants list: tiled
 *     attention == naive attention; llm-infer, "References": FlashAttention-2);
 *   - causal chunked prefill over a cached prefix (infer-lab, "Technique"
 *     table: chunked prefill; invariants: chunked == one-shot);
 *   - the 128-token sliding window (RustInfer, "Status": SWA operators with a
 *     128-token ring cache);
 *   - the merge of partial (o, lse) states (FlashAttention-2 work
 *     partitioning, llm-infer "References").
 *
 * Precision: attention runs in fp32 (the pages' correctness gate is an fp32
 * reference: llm-infer, "Results" and "How the Claims Are Checked"), with an
 * fp64 variant selected by `precision == 64` that bounds the fp32 oracle's own
 * rounding error.  Every sum runs in ascending index order; every product and
 * sum is a separately rounded operation (build with -ffp-contract=off).
 *
 * Readings of points the pages leave open:
 *   cache layout [num_blocks][Hkv][block_size][D], K and V in separate pools;
 *   query head h reads KV head h / (Hq / Hkv);
 *   RoPE is the half-split (NeoX) form over the whole head_dim, fp32, with a
 *   cos/sin table computed in double and rounded to fp32;
 *   the decode token sits at position context_len - 1;
 *   FP8 is OCP E4M3FN, stored = RNE-satfinite(x / scale), read = code * scale,
 *   quantised straight from the fp32 rotated value;
 *   window W keeps keys t with p - W < t <= p (W <= 0: no window);
 *   a query with no visible key yields o = 0, lse = -inf;
 *   lse is the natural-log sum of exp of the scaled logits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_KV_BF16 0
#define ORC_KV_FP8_E4M3 1

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 is the upper half of an IEEE binary32 word: widening is exact. */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even narrowing of binary32 to bf16.  NaN maps to the
 * canonical quiet NaN 0x7FFF with the sign kept. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FFFu);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    /* lower > half: round up; lower == half: round to even upper. */
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* a carry into the exponent is the correct result */
    return (uint16_t)upper;
}

/* ---------------------------------------------------------------- e4m3 --- */
/* OCP 8-bit floating point, E4M3FN: 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, NaN = S.1111.111, largest finite 448,
 * smallest subnormal 2^-9. */

float orc_e4m3_to_f32(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    float v;
    if (e == 0xF && m == 0x7) return s ? -NAN : NAN;
    if (e == 0)
        v = ldexpf((float)m, -9);            /* m/8 * 2^(1-7) */
    else
        v = ldexpf((float)(8 + m), e - 10);  /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Round-to-nearest-even encoding with saturation to +-448 (inf included);
 * NaN encodes as 0x7F / 0xFF. */
uint8_t orc_f32_to_e4m3(float x) {
    if (isnan(x)) return signbit(x) ? 0xFF : 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    /* exponent of the leading bit, clamped at the subnormal exponent -6 */
    int e2;
    frexp(a, &e2);               /* a = f * 2^e2, f in [0.5, 1) */
    int ex = e2 - 1;
    if (ex < -6) ex = -6;
    double quantum = ldexp(1.0, ex - 3);
    double n = nearbyint(a / quantum); /* a/quantum is exact; RNE to integer */
    double r = n * quantum;            /* rounded magnitude, exact */
    if (r >= 448.0) return (uint8_t)(sign | 0x7E);
    if (r == 0.0) return sign;
    frexp(r, &e2);
    int er = e2 - 1;
    if (er < -6) /* subnormal: r = m * 2^-9 */
        return (uint8_t)(sign | (uint8_t)(int)ldexp(r, 9));
    int m = (int)ldexp(r, 3 - er) - 8; /* r = (1 + m/8) * 2^er */
    return (uint8_t)(sign | (uint8_t)(((er + 7) << 3) | m));
}

/* ---------------------------------------------------------------- RoPE --- */

/* cos/sin table, fp32 [max_pos][rotary_dim/2][2] = (cos, sin) of
 * p * theta^(-2i/rotary_dim), computed in double and rounded once. */
void orc_rope_table(float theta, int32_t rotary_dim, int32_t max_pos, float *out) {
    int half = rotary_dim / 2;
    for (int p = 0; p < max_pos; ++p) {
        for (int i = 0; i < half; ++i) {
            double inv_freq = pow((double)theta, -(2.0 * (double)i) / (double)rotary_dim);
            double angle = (double)p * inv_freq;
            out[((size_t)p * half + i) * 2 + 0] = (float)cos(angle);
            out[((size_t)p * half + i) * 2 + 1] = (float)sin(angle);
        }
    }
}

/* Rotate one head vector (bf16 in, fp32 out) by the half-split rule
 *   x'[i]       = a*c - b*s
 *   x'[i + D/2] = b*c + a*s
 * with a = x[i], b = x[i + D/2]; each product and difference rounded. */
static void rope_rotate(const uint16_t *x, int D, const float *cs, float *outv) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        float a = orc_bf16_to_f32(x[i]);
        float b = orc_bf16_to_f32(x[i + half]);
        float c = cs[2 * i + 0];
        float s = cs[2 * i + 1];
        float ac = a * c;
        float bs = b * s;
        float bc = b * c;
        float as = a * s;
        outv[i] = ac - bs;
        outv[i + half] = bc + as;
    }
}

/* -------------------------------------------------------- append + RoPE --- */

/* Writes each new token's K and V into its slot of the paged cache and
 * rotates q in place.  Token i belongs to sequence token_to_seq[i] and sits
 * at position positions[i]; its slot is block block_tables[s][p / bs],
 * row p % bs -- or, with a ring of ring_blocks > 0 blocks per sequence (the
 * sliding-window cache of RustInfer's "Status"), block
 * block_tables[s][(p / bs) % ring_blocks].  K is rotated (when cos_sin != NULL) then rounded to bf16, or
 * divided by k_scale[h] and encoded as e4m3.  V is copied (bf16) or divided
 * by v_scale[h] and encoded.  Returns 0, or -1 on an out-of-range index (no
 * write happens for that token). */
int orc_append_rope(int32_t Hq, int32_t Hkv, int32_t D, int32_t bs, int32_t kv_dtype,
                    int64_t num_blocks, int32_t max_blocks_per_seq, int32_t ring_blocks,
                    void *k_cache, void *v_cache, const float *k_scale, const float *v_scale,
                    const int32_t *block_tables, int32_t num_seqs,
                    const int32_t *token_to_seq, const int32_t *positions, int32_t num_tokens,
                    const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_inout,
                    const float *cos_sin, int32_t max_pos) {
    int rc = 0;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)D);
    if (!tmp) return -2;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int32_t s = token_to_seq[i];
        int32_t p = positions[i];
        int32_t b = ring_blocks > 0 ? (p / bs) % ring_blocks : p / bs;
        if (s < 0 || s >= num_seqs || p < 0 || b >= max_blocks_per_seq ||
            (cos_sin && p >= max_pos)) { rc = -1; continue; }
        int32_t blk = block_tables[(size_t)s * max_blocks_per_seq + b];
        if (blk < 0 || (int64_t)blk >= num_blocks) { rc = -1; continue; }
        int32_t slot = p % bs;
        const float *cs = cos_sin ? cos_sin + (size_t)p * (D / 2) * 2 : NULL;
        for (int32_t h = 0; h < Hkv; ++h) {
            size_t src = ((size_t)i * Hkv + h) * D;
            size_t dst = (((size_t)blk * Hkv + h) * bs + slot) * D;
            const uint16_t *kx = k_new + src;
            const uint16_t *vx = v_new + src;
            if (cs) rope_rotate(kx, D, cs, tmp);
            else for (int d = 0; d < D; ++d) tmp[d] = orc_bf16_to_f32(kx[d]);
            if (kv_dtype == ORC_KV_BF16) {
                uint16_t *kc = (uint16_t *)k_cache + dst;
                uint16_t *vc = (uint16_t *)v_cache + dst;
                for (int d = 0; d < D; ++d) kc[d] = orc_f32_to_bf16(tmp[d]);
                for (int d = 0; d < D; ++d) vc[d] = vx[d];
            } else {
                uint8_t *kc = (uint8_t *)k_cache + dst;
                uint8_t *vc = (uint8_t *)v_cache + dst;
                for (int d = 0; d < D; ++d) kc[d] = orc_f32_to_e4m3(tmp[d] / k_scale[h]);
                for (int d = 0; d < D; ++d)
                    vc[d] = orc_f32_to_e4m3(orc_bf16_to_f32(vx[d]) / v_scale[h]);
            }
        }
        if (q_inout && cs) {
            for (int32_t h = 0; h < Hq; ++h) {
                uint16_t *qx = q_inout + ((size_t)i * Hq + h) * D;
                rope_rotate(qx, D, cs, tmp);
                for (int d = 0; d < D; ++d) qx[d] = orc_f32_to_bf16(tmp[d]);
            }
        }
    }
    free(tmp);
    return rc;
}

/* ------------------------------------------------------------ block copy --- */

/* Copy-on-write of paged blocks: block dst[i] of a pool receives the bytes
 * of block src[i] (every head, every row).  block_bytes = Hkv*bs*D*elem.
 * Returns 0, or -1 if an id is out of range (that pair is skipped). */
int orc_copy_blocks(void *cache, int64_t num_blocks, int64_t block_bytes, const int32_t *src,
                    const int32_t *dst, int32_t num_pairs) {
    int rc = 0;
    for (int32_t i = 0; i < num_pairs; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
            rc = -1;
            continue;
        }
        memcpy((uint8_t *)cache + (size_t)dst[i] * block_bytes,
               (const uint8_t *)cache + (size_t)src[i] * block_bytes, (size_t)block_bytes);
    }
    return rc;
}

/* --------------------------------------------------------------- gather --- */

/* out[cu[s] + t][h][:] = cache[block_tables[s][t / bs]][h][t % bs][:] for
 * t < lens[s]; a byte copy (elem_bytes = 2 for bf16, 1 for e4m3). */
int orc_gather_kv(int32_t Hkv, int32_t D, int32_t bs, int32_t elem_bytes, int64_t num_blocks,
                  int32_t max_blocks_per_seq, const void *cache, const int32_t *block_tables,
                  const int32_t *lens, int32_t num_seqs, void *out) {
    size_t row = (size_t)D * elem_bytes;
    size_t o = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        for (int32_t t = 0; t < lens[s]; ++t) {
            if (t / bs >= max_blocks_per_seq) return -1;
            int32_t blk = block_tables[(size_t)s * max_blocks_per_seq + t / bs];
            if (blk < 0 || (int64_t)blk >= num_blocks) return -1;
            for (int32_t h = 0; h < Hkv; ++h) {
                const uint8_t *src = (const uint8_t *)cache +
                                     (((size_t)blk * Hkv + h) * bs + (t % bs)) * row;
                memcpy((uint8_t *)out + (o * Hkv + h) * row, src, row);
            }
            ++o;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ attention --- */

typedef struct {
    int32_t Hq, Hkv, D, bs, kv_dtype, max_blocks_per_seq;
    int64_t num_blocks;
    const void *k_cache, *v_cache;
    const float *k_scale, *v_scale;
    const int32_t *block_tables;
    int32_t num_seqs;
    const int32_t *qo_indptr, *kv_lens;
    const uint16_t *q;
    float sm_scale;
    int32_t causal, window, precision;
    int32_t ring_blocks;     /* > 0: key t sits in table entry (t / bs) % ring_blocks */
    const float *sinks;      /* nullable: per query head sink logit */
    float *out, *lse;
    const int32_t *tok_seq; /* query token -> sequence, filled by the caller */
    int64_t units;          /* num_q_tokens * Hq */
    int64_t begin, end;
    int err;
} attn_job;

/* K or V element d of key t of sequence s, KV head h, as fp32 (dequantised
 * with the per-head scale for e4m3). */
static float kv_elem(const attn_job *J, const void *cache, const float *scale,
                     int32_t s, int32_t t, int32_t h, int32_t d, int *err) {
    int32_t b = J->ring_blocks > 0 ? (t / J->bs) % J->ring_blocks : t / J->bs;
    int32_t blk = J->block_tables[(size_t)s * J->max_blocks_per_seq + b];
    if (blk < 0 || (int64_t)blk >= J->num_blocks) { *err = 1; return 0.0f; }
    size_t idx = (((size_t)blk * J->Hkv + h) * J->bs + (t % J->bs)) * J->D + d;
    if (J->kv_dtype == ORC_KV_BF16) return orc_bf16_to_f32(((const uint16_t *)cache)[idx]);
    return orc_e4m3_to_f32(((const uint8_t *)cache)[idx]) * scale[h];
}

/* One (query token, query head) output: the plain softmax-attention
 * definition over the keys the mask leaves visible.
 *   l_t = sm_scale * sum_d q[d] k_t[d]
 *   m = max_t l_t,  e_t = exp(l_t - m),  L = sum_t e_t
 *   o = (sum_t e_t v_t) / L,  lse = m + ln L
 * With a sink logit s for the head (a softmax entry whose value is zero):
 *   m = max(s, max_t l_t),  L = exp(s - m) + sum_t e_t.                      */
static void attend_one_f32(attn_job *J, int64_t unit, float *logit, float *acc) {
    int32_t i = (int32_t)(unit / J->Hq);
    int32_t h = (int32_t)(unit % J->Hq);
    int32_t s = J->tok_seq[i];
    int32_t G = J->Hq / J->Hkv;
    int32_t kvh = h / G;
    int32_t kv_len = J->kv_lens[s];
    int32_t q_len = J->qo_indptr[s + 1] - J->qo_indptr[s];
    int32_t pos = kv_len - q_len + (i - J->qo_indptr[s]);
    int32_t hi = J->causal ? pos : kv_len - 1;  /* last visible key */
    if (hi > kv_len - 1) hi = kv_len - 1;
    int32_t lo = 0;
    if (J->window > 0 && pos - J->window + 1 > lo) lo = pos - J->window + 1;
    const uint16_t *qv = J->q + ((size_t)i * J->Hq + h) * J->D;
    float *o = J->out + ((size_t)i * J->Hq + h) * J->D;
    int err = 0;
    const float sink = J->sinks ? J->sinks[h] : -INFINITY;
    if (hi < lo) {
        for (int d = 0; d < J->D; ++d) o[d] = 0.0f;
        if (J->lse) J->lse[(size_t)i * J->Hq + h] = sink;
        return;
    }
    int32_t n = hi - lo + 1;
    for (int32_t t = 0; t < n; ++t) {
        float dot = 0.0f;
        for (int d = 0; d < J->D; ++d)
            dot += orc_bf16_to_f32(qv[d]) * kv_elem(J, J->k_cache, J->k_scale, s, lo + t, kvh, d, &err);
        logit[t] = J->sm_scale * dot;
    }
    float m = logit[0];
    for (int32_t t = 1; t < n; ++t) if (logit[t] > m) m = logit[t];
    if (sink > m) m = sink;
    float L = sink == -INFINITY ? 0.0f : expf(sink - m);
    for (int32_t t = 0; t < n; ++t) { logit[t] = expf(logit[t] - m); L += logit[t]; }
    for (int d = 0; d < J->D; ++d) acc[d] = 0.0f;
    for (int32_t t = 0; t < n; ++t)
        for (int d = 0; d < J->D; ++d)
            acc[d] += logit[t] * kv_elem(J, J->v_cache, J->v_scale, s, lo + t, kvh, d, &err);
    for (int d = 0; d < J->D; ++d) o[d] = acc[d] / L;
    if (J->lse) J->lse[(size_t)i * J->Hq + h] = m + logf(L);
    if (err) J->err = 1;
}

/* The same definition carried out in double. */
static void attend_one_f64(attn_job *J, int64_t unit, double *logit, double *acc) {
    int32_t i = (int32_t)(unit / J->Hq);
    int32_t h = (int32_t)(unit % J->Hq);
    int32_t s = J->tok_seq[i];
    int32_t G = J->Hq / J->Hkv;
    int32_t kvh = h / G;
    int32_t kv_len = J->kv_lens[s];
    int32_t q_len = J->qo_indptr[s + 1] - J->qo_indptr[s];
    int32_t pos = kv_len - q_len + (i - J->qo_indptr[s]);
    int32_t hi = J->causal ? pos : kv_len - 1;
    if (hi > kv_len - 1) hi = kv_len - 1;
    int32_t lo = 0;
    if (J->window > 0 && pos - J->window + 1 > lo) lo = pos - J->window + 1;
    const uint16_t *qv = J->q + ((size_t)i * J->Hq + h) * J->D;
    float *o = J->out + ((size_t)i * J->Hq + h) * J->D;
    int err = 0;
    const double sink = J->sinks ? (double)J->sinks[h] : -INFINITY;
    if (hi < lo) {
        for (int d = 0; d < J->D; ++d) o[d] = 0.0f;
        if (J->lse) J->lse[(size_t)i * J->Hq + h] = (float)sink;
        return;
    }
    int32_t n = hi - lo + 1;
    for (int32_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int d = 0; d < J->D; ++d)
            dot += (double)orc_bf16_to_f32(qv[d]) *
                   (double)kv_elem(J, J->k_cache, J->k_scale, s, lo + t, kvh, d, &err);
        logit[t] = (double)J->sm_scale * dot;
    }
    double m = logit[0];
    for (int32_t t = 1; t < n; ++t) if (logit[t] > m) m = logit[t];
    if (sink > m) m = sink;
    double L = sink == -INFINITY ? 0.0 : exp(sink - m);
    for (int32_t t = 0; t < n; ++t) { logit[t] = exp(logit[t] - m); L += logit[t]; }
    for (int d = 0; d < J->D; ++d) acc[d] = 0.0;
    for (int32_t t = 0; t < n; ++t)
        for (int d = 0; d < J->D; ++d)
            acc[d] += logit[t] * (double)kv_elem(J, J->v_cache, J->v_scale, s, lo + t, kvh, d, &err);
    for (int d = 0; d < J->D; ++d) o[d] = (float)(acc[d] / L);
    if (J->lse) J->lse[(size_t)i * J->Hq + h] = (float)(m + log(L));
    if (err) J->err = 1;
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    int32_t max_len = 0;
    for (int32_t s = 0; s < J->num_seqs; ++s) if (J->kv_lens[s] > max_len) max_len = J->kv_lens[s];
    /* a causal window holds at most W keys; without causality a query's
     * range [p - W + 1, kv_len) can be longer, so only causal windows cap it */
    if (J->causal && J->window > 0 && J->window < max_len) max_len = J->window;
    size_t n = (size_t)(max_len > 0 ? max_len : 1);
    if (J->precision == 64) {
        double *logit = (double *)malloc(sizeof(double) * n);
        double *acc = (double *)malloc(sizeof(double) * (size_t)J->D);
        if (!logit || !acc) { J->err = 2; free(logit); free(acc); return NULL; }
        for (int64_t u = J->begin; u < J->end; ++u) attend_one_f64(J, u, logit, acc);
        free(logit); free(acc);
    } else {
        float *logit = (float *)malloc(sizeof(float) * n);
        float *acc = (float *)malloc(sizeof(float) * (size_t)J->D);
        if (!logit || !acc) { J->err = 2; free(logit); free(acc); return NULL; }
        for (int64_t u = J->begin; u < J->end; ++u) attend_one_f32(J, u, logit, acc);
        free(logit); free(acc);
    }
    return NULL;
}

/* Ragged attention over the paged cache.  Sequence s owns query tokens
 * [qo_indptr[s], qo_indptr[s+1]) and kv_lens[s] cached keys; its query i sits
 * at position kv_lens[s] - q_len + (i - qo_indptr[s]).  Decode is the case
 * q_len = 1 for every sequence.  q: bf16 [T][Hq][D]; out: fp32 [T][Hq][D];
 * lse (nullable): fp32 [T][Hq].  ring_blocks > 0: the sequence's cache is a
 * ring of that many blocks (key t in table entry (t / bs) % ring_blocks); a
 * window is then required and its keys must fit the ring.  sinks (nullable):
 * fp32 [Hq] sink logits.  Units (token, head) are spread over nthreads
 * threads; the result does not depend on nthreads.
 * Returns 0; -1 on a bad argument; 1 if a block id was out of range. */
int orc_paged_attention(int32_t Hq, int32_t Hkv, int32_t D, int32_t bs, int32_t kv_dtype,
                        int64_t num_blocks, int32_t max_blocks_per_seq,
                        const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_tables, int32_t num_seqs,
                        const int32_t *qo_indptr, const int32_t *kv_lens,
                        const uint16_t *q, float sm_scale, int32_t causal, int32_t window,
                        int32_t ring_blocks, const float *sinks,
                        float *out, float *lse, int32_t precision, int32_t nthreads) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || bs <= 0 || num_seqs < 0) return -1;
    if (ring_blocks < 0 || ring_blocks > max_blocks_per_seq) return -1;
    /* a window spans at most (window - 1 + bs - 1) / bs + 1 blocks */
    if (ring_blocks > 0 && (window <= 0 || (window - 1 + bs - 1) / bs + 1 > ring_blocks)) return -1;
    int32_t T = qo_indptr[num_seqs];
    for (int32_t s = 0; s < num_seqs; ++s) {
        if (qo_indptr[s + 1] < qo_indptr[s]) return -1;
        if (kv_lens[s] < 0 || (ring_blocks == 0 && (kv_lens[s] + bs - 1) / bs > max_blocks_per_seq))
            return -1;
    }
    int32_t *tok_seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!tok_seq) return -2;
    for (int32_t s = 0; s < num_seqs; ++s)
        for (int32_t i = qo_indptr[s]; i < qo_indptr[s + 1]; ++i) tok_seq[i] = s;
    if (nthreads < 1) nthreads = 1;
    int64_t units = (int64_t)T * Hq;
    if (nthreads > units) nthreads = (int32_t)(units > 0 ? units : 1);
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); free(tok_seq); return -2; }
    for (int32_t w = 0; w < nthreads; ++w) {
        attn_job *J = &jobs[w];
        J->Hq = Hq; J->Hkv = Hkv; J->D = D; J->bs = bs; J->kv_dtype = kv_dtype;
        J->max_blocks_per_seq = max_blocks_per_seq; J->num_blocks = num_blocks;
        J->k_cache = k_cache; J->v_cache = v_cache; J->k_scale = k_scale; J->v_scale = v_scale;
        J->block_tables = block_tables; J->num_seqs = num_seqs;
        J->qo_indptr = qo_indptr; J->kv_lens = kv_lens; J->q = q; J->sm_scale = sm_scale;
        J->causal = causal; J->window = window; J->precision = precision;
        J->ring_blocks = ring_blocks; J->sinks = sinks;
        J->out = out; J->lse = lse; J->tok_seq = tok_seq; J->units = units;
        J->begin = units * w / nthreads;
        J->end = units * (w + 1) / nthreads;
    }
    int rc = 0;
    if (nthreads == 1) {
        attn_worker(&jobs[0]);
    } else {
        int32_t started = 0;
        for (int32_t w = 0; w < nthreads; ++w) {
            if (pthread_create(&th[w], NULL, attn_worker, &jobs[w]) != 0) break;
            ++started;
        }
        for (int32_t w = started; w < nthreads; ++w) attn_worker(&jobs[w]);
        for (int32_t w = 0; w < started; ++w) pthread_join(th[w], NULL);
    }
    for (int32_t w = 0; w < nthreads; ++w) {
        if (jobs[w].err == 2) rc = -2;
        else if (jobs[w].err && rc == 0) rc = 1;
    }
    free(jobs); free(th); free(tok_seq);
    return rc;
}

/* ---------------------------------------------------------------- merge --- */

/* Merge of P partial attention states over disjoint key sets:
 *   M = max_i lse_i,  w_i = exp(lse_i - M)
 *   o = sum_i w_i o_i / sum_i w_i,  lse = M + ln sum_i w_i
 * A part with lse = -inf has weight 0; if every part is empty the result is
 * o = 0, lse = -inf.  o_parts: fp32 [P][rows][H][D]; lse_parts [P][rows][H];
 * out fp32 [rows][H][D]; lse_out (nullable) [rows][H]. */
void orc_merge_states(const float *o_parts, const float *lse_parts, int32_t P, int32_t rows,
                      int32_t H, int32_t D, float *out, float *lse_out) {
    size_t RH = (size_t)rows * H;
    for (size_t r = 0; r < RH; ++r) {
        float M = -INFINITY;
        for (int32_t i = 0; i < P; ++i)
            if (lse_parts[(size_t)i * RH + r] > M) M = lse_parts[(size_t)i * RH + r];
        float *o = out + r * D;
        if (M == -INFINITY) {
            for (int d = 0; d < D; ++d) o[d] = 0.0f;
            if (lse_out) lse_out[r] = -INFINITY;
            continue;
        }
        float W = 0.0f;
        for (int d = 0; d < D; ++d) o[d] = 0.0f;
        for (int32_t i = 0; i < P; ++i) {
            if (lse_parts[(size_t)i * RH + r] == -INFINITY) continue; /* empty part */
            float w = expf(lse_parts[(size_t)i * RH + r] - M);
            W += w;
            const float *oi = o_parts + ((size_t)i * RH + r) * D;
            for (int d = 0; d < D; ++d) o[d] += w * oi[d];
        }
        for (int d = 0; d < D; ++d) o[d] = o[d] / W;
        if (lse_out) lse_out[r] = M + logf(W);
    }
}

/* ------------------------------------------------ array conversions ------ */
/* Element-wise loops over the scalar routines above, for bulk checks. */

void orc_bf16_to_f32_array(const uint16_t *in, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}

void orc_f32_to_bf16_array(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

void orc_e4m3_to_f32_array(const uint8_t *in, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f32(in[i]);
}

void orc_f32_to_e4m3_array(const float *in, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(in[i]);
}
