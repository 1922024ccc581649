/*
 * pkv.h -- C ABI of libpkv: attention over a paged KV cache, hand-written
 * CUDA for one GB300 (sm_103a).
 *
 * The operations follow four serving engines' descriptions of the same hot
 * path (InferX; infer-lab; llm-infer; RustInfer):
 *   - a paged KV cache: fixed-size blocks and per-sequence block tables
 *     (infer-lab, "Technique" table, PagedAttention; llm-infer, "What It
 *     Does"; InferX, "Status" and roadmap M3);
 *   - the KV write of each new token fused with RoPE (llm-infer, "What It
 *     Does": graphs capture the KV writes, RMSNorm and RoPE fused);
 *   - GQA decode attention with an online softmax, split across KV chunks
 *     and merged (llm-infer, "References": FlashAttention-2 work
 *     partitioning; infer-lab, "Strategy" table: tiled/online softmax);
 *   - causal, ragged, chunked prefill over cached prefixes (infer-lab,
 *     "Technique" table: chunked prefill; llm-infer, "What It Does": ragged
 *     batched prefill);
 *   - an FP8 e4m3 KV cache with per-head scales (InferX, "The kernels
 *     underneath", M8) and a 128-token sliding window (RustInfer, "Status").
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer unless its comment says "host".
 *   - The caller owns every buffer (caches, tables, q/out, cos/sin table,
 *     workspace).  The library allocates no device memory on any call; it
 *     caches CUDA tensor-map descriptors, which are host data.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream); no call synchronises the device.
 *   - Arguments are validated on the host before any launch; a failed check
 *     returns its status and touches no device memory.  pkv_last_error()
 *     then describes the failure (thread-local, valid until the next call).
 *   - Device-side checks (a block id outside [0, num_blocks), a position
 *     outside the table, a wait that ran out) never trap: the offending
 *     access is skipped or clamped and a bit is set in the device error word
 *     read by pkv_device_errors().
 *
 * Cache layout (one pool for K, one for V): [num_blocks][Hkv][block_size][D]
 * of bf16 or e4m3 bytes.  Token t of sequence s lives in block
 * block_tables[s * max_blocks_per_seq + t / block_size], row
 * t % block_size.  Query head h reads KV head h / (Hq / Hkv).
 * q and out are [tokens][Hq][D] bf16; lse is [tokens][Hq] fp32, natural log.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent sizes, bad lengths */
    PKV_ERR_UNSUPPORTED = 2,  /* head_dim, block_size, dtype or group size not built */
    PKV_ERR_WORKSPACE = 3,    /* workspace null, too small or misaligned */
    PKV_ERR_CUDA = 4          /* a CUDA runtime/driver call or launch failed */
} pkv_status;

typedef enum { PKV_KV_BF16 = 0, PKV_KV_FP8_E4M3 = 1 } pkv_kv_dtype;

/* Device error word bits (pkv_device_errors). */
#define PKV_DEVERR_BLOCK_ID 0x1u  /* a block id outside [0, num_blocks): access skipped */
#define PKV_DEVERR_POSITION 0x2u  /* a position/sequence index outside its table: skipped */
#define PKV_DEVERR_TIMEOUT 0x4u   /* a bounded wait gave up: that output is invalid */
#define PKV_DEVERR_LENGTH 0x8u    /* a length beyond the table capacity: clamped */

/* Shape of one paged KV pool pair (K and V share it).
 * Supported: head_dim 64 or 128; block_size 16; num_q_heads a multiple of
 * num_kv_heads with group size num_q_heads / num_kv_heads <= 16.
 * ring_blocks > 0 makes every sequence's cache a ring of that many blocks, as
 * for a sliding-window layer (RustInfer, "Status": SWA with a 128-token ring
 * cache): token p lives in block block_tables[s][(p / block_size) % ring_blocks],
 * so a sequence's window of W keys needs ring_blocks >= ceil((W - 1) / 16) + 1
 * (9 for W = 128) however long it grows.  Append and decode (with a window)
 * honour it; prefill, gather and cascade decode refuse a ring (PKV_ERR_UNSUPPORTED). */
typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t kv_dtype;            /* pkv_kv_dtype */
    int32_t max_blocks_per_seq;  /* row length of block_tables (int32 [num_seqs][this]) */
    int64_t num_blocks;          /* blocks in each pool */
    int32_t ring_blocks;         /* 0: linear tables; > 0: ring of this many blocks (<= max_blocks_per_seq) */
    uint32_t flags;              /* PKV_DESC_* bits; 0 for none */
} pkv_cache_desc;

/* pkv_cache_desc.flags.
 * PKV_DESC_PREFETCH_KV: a promise about the stream the calls run on: the
 *   kernel launched just before a decode call (pkv_decode_attention, _step,
 *   _static) writes none of the K/V rows, block-table entries or context
 *   lengths that call reads -- it may write q, k_new and v_new, as the layer's
 *   QKV projection does.  The decode kernel then reads the lengths and block
 *   ids and starts its first K/V loads while that kernel drains (programmatic
 *   dependent launch, llm-infer "What It Does": CUDA-graphed decode), and
 *   waits for it before it reads q, k_new or v_new and before any write.
 *   Without the promise (the default) nothing is read before that wait.  A
 *   call whose predecessor breaks the promise may read stale K/V rows. */
#define PKV_DESC_PREFETCH_KV 0x1u
/* PKV_DESC_INDEPENDENT: a stronger promise: the kernel launched just before a
 *   decode call reads and writes nothing the call reads or writes -- as when
 *   the call is the decode half of one layer's mixed step and the prefill half
 *   ran just before it (both read the same QKV projection's output, different
 *   sequences' blocks, different outputs).  The decode kernel then runs
 *   without waiting for that kernel (its CTAs take the SMs the prefill's last
 *   CTAs leave idle) and waits for it only at its end, so kernels launched
 *   after the call still see both.  Implies PKV_DESC_PREFETCH_KV.
 * Both promises are about the kernel just before the call.  Kernels launched
 * earlier are complete by the time the call starts as long as that kernel
 * lets its dependents start only once its own predecessor has completed, as
 * every kernel of this library does (and as any kernel launched without
 * programmatic stream serialization does by construction). */
#define PKV_DESC_INDEPENDENT 0x2u

/* Bytes of one pool (K or V): num_blocks * Hkv * block_size * head_dim * elem.
 * Host only; 0 for an invalid desc. */
uint64_t pkv_cache_bytes(const pkv_cache_desc *desc);

/* ---- a1: fused KV append + RoPE (llm-infer, "What It Does") ------------
 * For each new token i (0 <= i < num_tokens): s = token_to_seq[i],
 * p = positions[i]; slot = block block_tables[s][p / block_size] (entry
 * (p / block_size) % ring_blocks with a ring), row p % block_size.  For every KV head h:
 *   K row = RoPE(k_new[i][h], p) rounded to bf16 (RNE), or for e4m3
 *           RNE-satfinite(RoPE(k_new[i][h], p) / k_scale[h]);
 *   V row = v_new[i][h] copied, or RNE-satfinite(v_new[i][h] / v_scale[h]).
 * q_inout[i][h'] is rotated in place for every query head (skipped if NULL).
 * RoPE is the half-split form over the whole head: with a = x[j],
 * b = x[j + D/2], c/s = rope_cos_sin[p][j][0/1]:
 *   x'[j] = a*c - b*s,  x'[j + D/2] = b*c + a*s   (fp32, each op rounded).
 * rope_cos_sin == NULL: no rotation (plain append).
 *   k_cache, v_cache : pools, written.   k_scale, v_scale: fp32 [Hkv], e4m3 only.
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq].
 *   token_to_seq, positions : int32 [num_tokens].
 *   k_new, v_new     : bf16 [num_tokens][Hkv][D].  q_inout: bf16 [num_tokens][Hq][D].
 *   rope_cos_sin     : fp32 [rope_max_pos][D/2][2] (pkv_rope_cos_sin_table).
 * Two tokens must not target the same slot in one call. */
pkv_status pkv_append_rope(const pkv_cache_desc *desc, void *k_cache, void *v_cache,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_tables, int32_t num_seqs,
                           const int32_t *token_to_seq, const int32_t *positions,
                           int32_t num_tokens, const void *k_new, const void *v_new,
                           void *q_inout, const float *rope_cos_sin, int32_t rope_max_pos,
                           pkv_stream_t stream);

/* Host: fill host_out (fp32 [max_pos][rotary_dim/2][2]) with (cos, sin) of
 * p * theta^(-2j/rotary_dim), computed in double and rounded once to fp32. */
pkv_status pkv_rope_cos_sin_table(float theta, int32_t rotary_dim, int32_t max_pos,
                                  float *host_out);

/* ---- a2: block-table gather (infer-lab, "Technique" table) -------------
 * out[cu_context_lens[s] + t][h][:] = cache[bt[s][t / bs]][h][t % bs][:] for
 * t < context_lens[s]: a byte-exact copy of one pool into contiguous
 * [total_tokens][Hkv][D] (bf16 or e4m3 bytes).  cu_context_lens: int32
 * [num_seqs + 1], prefix sums of context_lens; total_tokens its last entry
 * (host value).  The decode and prefill kernels do this gather themselves,
 * block by block, through TMA; this export exists so the addressing can be
 * checked bit for bit. */
pkv_status pkv_gather_kv(const pkv_cache_desc *desc, const void *cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         const int32_t *cu_context_lens, int32_t num_seqs,
                         int64_t total_tokens, void *out, pkv_stream_t stream);

/* ---- copy-on-write of shared blocks (infer-lab, "Technique" table:
 * PagedAttention refcounting and copy-on-write; llm-infer, "What It Does") --
 * For i < num_pairs, block dst_blocks[i] of both pools receives the bytes of
 * block src_blocks[i] (every head, every row).  src_blocks, dst_blocks: int32
 * [num_pairs].  dst ids must be distinct and must not appear among the src
 * ids of the same call.  An id outside [0, num_blocks) skips that pair and
 * sets PKV_DEVERR_BLOCK_ID. */
pkv_status pkv_copy_blocks(const pkv_cache_desc *desc, void *k_cache, void *v_cache,
                           const int32_t *src_blocks, const int32_t *dst_blocks, int32_t num_pairs,
                           pkv_stream_t stream);

/* ---- a3-a7: split-KV GQA decode (FlashAttention-2 partitioning) ---------
 * One query token per sequence, at position context_lens[s] - 1 (the new
 * token, already appended).  For query head h, KV head h / G:
 *   o = softmax(sm_scale * q k^T) v over the visible keys, lse = ln sum exp.
 * Visible keys: t < context_lens[s]; with window > 0 also
 * t > context_lens[s] - 1 - window.  e4m3 pools read k = code * k_scale[h],
 * v = code * v_scale[h].  With sinks (RustInfer, "Status": SWA operators
 * with attention sinks) query head h has a sink logit sinks[h] that joins
 * the softmax with a zero value: o = sum_t e^{l_t} v_t / (e^{sinks[h]} +
 * sum_t e^{l_t}), lse = ln(e^{sinks[h]} + sum_t e^{l_t}).
 * The KV range of each (sequence, KV head) is cut into chunks of whole
 * blocks (pkv_decode_plan); every chunk runs as one CTA whose warps share
 * the G query heads of the group, and the chunks' partial (o, lse) states
 * merge in the same launch: with 2-4 chunks inside a thread-block cluster
 * (distributed shared memory), with more through the workspace, where the
 * last chunk to finish merges them.
 *   q        : bf16 [num_seqs][Hq][D].      out: bf16 [num_seqs][Hq][D].
 *   lse_out  : fp32 [num_seqs][Hq], nullable.
 *   context_lens : int32 [num_seqs], each in [1, max_blocks_per_seq*bs]
 *              (any length >= 1 with a ring cache).
 *   max_context_len : host, >= every context_lens[s]; sizes the plan.
 *   window   : <= 0 for full attention; required (> 0, and covered by the
 *              ring) when desc->ring_blocks > 0.
 *   sinks    : fp32 [Hq] sink logits in the units of sm_scale * q.k, or NULL.
 *   chunk_blocks : blocks per chunk; 0 lets the planner choose
 *              (pkv_decode_plan), else 1..256 (1..128 for e4m3 pools).  A
 *              context is cut into at most 512 chunks, so the visible keys of
 *              one sequence are limited to 512 x 256 x 16 (bf16) or
 *              512 x 128 x 16 (e4m3) tokens: PKV_ERR_UNSUPPORTED beyond.
 *   workspace: >= pkv_decode_workspace_size(...) bytes, 256-byte aligned,
 *              zero-filled before its first use; every call leaves it
 *              zeroed again.  Calls that share a workspace must not overlap
 *              on the GPU.
 * Host-resident per-step arrays: with unified addressing (a GB300 and its
 * Grace host), q, block_tables, context_lens, k_scale, v_scale, sinks, out
 * and lse_out -- and k_new, v_new of pkv_decode_step -- may be pinned
 * (page-locked) host memory.  The kernel then reads and writes them over the
 * host link itself, so a step needs no separate copies; the results are the
 * same bytes.  The pools, the workspace and rope_cos_sin stay in device
 * memory. */
pkv_status pkv_decode_attention(const pkv_cache_desc *desc, const void *q,
                                const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_tables, const int32_t *context_lens,
                                int32_t num_seqs, int32_t max_context_len, float sm_scale,
                                int32_t window, const float *sinks, int32_t chunk_blocks,
                                void *out, float *lse_out, void *workspace,
                                size_t workspace_bytes, pkv_stream_t stream);

/* ---- a1 + a3-a7 fused: one decode step of one layer (llm-infer, "What It
 * Does": KV writes and fused RoPE inside the decode step).  Equal, bit for
 * bit in the cache and in out / lse, to
 *   pkv_append_rope(token_to_seq[s] = s, positions[s] = context_lens[s] - 1,
 *                   k_new, v_new, q_inout = a copy of q, rope_cos_sin)
 * followed by pkv_decode_attention over that rotated copy -- in one launch:
 * the CTA that loads a sequence's last block writes the new K/V rows into it
 * first, and every CTA rotates its own query rows.  q itself is only read
 * (not rotated in place).
 *   k_new, v_new : bf16 [num_seqs][Hkv][D], the new token's K (before RoPE)
 *                  and V; context_lens[s] already counts that token.
 *   rope_cos_sin : fp32 [rope_max_pos][D/2][2] (pkv_rope_cos_sin_table), or
 *                  NULL (no rotation); rope_max_pos >= max_context_len.
 *   k_cache, v_cache : written (one row per sequence and KV head), then read.
 * A sequence with context_lens[s] == 0 appends nothing.  Two sequences'
 * new tokens must not share a slot.  Every other argument, the workspace
 * (pkv_decode_workspace_size) and the errors are those of
 * pkv_decode_attention. */
pkv_status pkv_decode_step(const pkv_cache_desc *desc, const void *q, const void *k_new,
                           const void *v_new, const float *rope_cos_sin, int32_t rope_max_pos,
                           void *k_cache, void *v_cache, const float *k_scale,
                           const float *v_scale, const int32_t *block_tables,
                           const int32_t *context_lens, int32_t num_seqs,
                           int32_t max_context_len, float sm_scale, int32_t window,
                           const float *sinks, int32_t chunk_blocks, void *out, float *lse_out,
                           void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Host: workspace bytes pkv_decode_attention needs for this shape and
 * chunk_blocks (0 = planned; planning uses the current device's SM count).
 * 0 when no workspace is needed (every sequence fits one chunk) or the
 * arguments are invalid. */
size_t pkv_decode_workspace_size(const pkv_cache_desc *desc, int32_t num_seqs,
                                 int32_t max_context_len, int32_t window, int32_t chunk_blocks);

/* ---- a4: the split planner (InferX, "Measured": a kernel launched with too
 * few CTAs cost 3.9x).  Host only.  Chooses the chunk length in whole blocks
 * so that the (sequence, KV head, chunk) CTAs fill the GPU several times
 * over; each sequence then has ceil(visible blocks / chunk) chunks.
 *   num_sms: SM count to plan for (<= 0: the current device's). */
pkv_status pkv_decode_plan(const pkv_cache_desc *desc, int32_t num_seqs,
                           int32_t max_context_len, int32_t window, int32_t num_sms,
                           int32_t *chunk_blocks_out, int32_t *max_splits_out);

/* ---- a8: ragged causal chunked prefill (infer-lab, chunked prefill) -----
 * Sequence s owns query tokens [qo_indptr[s], qo_indptr[s+1]) of q and
 * kv_lens[s] cached keys, its own chunk's K/V already appended; query i sits
 * at position kv_lens[s] - q_len + (i - qo_indptr[s]) and, with causal != 0,
 * sees keys t <= that position (window > 0: also t > position - window).
 *   q, out   : bf16 [total_q_tokens][Hq][D].  lse_out: fp32, nullable.
 *   qo_indptr: int32 [num_seqs + 1] (device).  kv_lens: int32 [num_seqs].
 *   qo_indptr_host, kv_lens_host: host copies (nullable, used for planning
 *              and validation only; they must match the device arrays).  With
 *              qo_indptr_host, a batch whose every sequence has at most 64
 *              query rows (q_len * Hq / Hkv: speculative verify, infer-lab
 *              "Technique" table) runs a decode-shaped kernel (mma.sync rows,
 *              KV cut into <= 4 chunks merged in a thread-block cluster);
 *              larger ones run the tcgen05 prefill.  kv_lens_host, when given,
 *              sizes that plan and orders the tcgen05 launch by work; without
 *              it the plan assumes full tables.
 *   k_scale, v_scale: fp32 [Hkv], e4m3 pools only (else NULL): k = code * k_scale[h],
 *              v = code * v_scale[h] (InferX, "The kernels underneath": FP8 KV cache).
 *   workspace: unused (may be NULL; pkv_prefill_workspace_size returns 0).
 *              Over e4m3 pools both kernels read the codes and convert them
 *              exactly on chip: the tcgen05 kernel into f16 tiles in shared
 *              memory, the short-query kernel into f16 MMA fragments; the
 *              MMAs are f16 with q rounded to f16 (exact for |q| in
 *              [2^-14, 65504]) and P in f16.
 * No ring cache (PKV_ERR_UNSUPPORTED): a ring takes pkv_prefill_ring_commit. */
pkv_status pkv_prefill_attention_ragged(const pkv_cache_desc *desc, const void *q,
                                        const int32_t *qo_indptr, const void *k_cache,
                                        const void *v_cache, const float *k_scale,
                                        const float *v_scale, const int32_t *block_tables,
                                        const int32_t *kv_lens, int32_t num_seqs,
                                        int32_t total_q_tokens, const int32_t *qo_indptr_host,
                                        const int32_t *kv_lens_host, float sm_scale,
                                        int32_t causal, int32_t window, void *out,
                                        float *lse_out, void *workspace,
                                        size_t workspace_bytes, pkv_stream_t stream);

/* ---- f4: ragged prefill over a sliding-window ring cache, with the cache
 * commit (RustInfer, "Status": Tensor Core prefill over full or chunked
 * inputs followed by a stream-ordered cache commit; SWA with a 128-token
 * ring cache).  desc->ring_blocks = R > 0: position p of sequence s lives in
 * table entry (p / 16) % R.  Sequence s brings q_len = qo_indptr[s+1] -
 * qo_indptr[s] new tokens at positions [kv_len - q_len, kv_len); the keys
 * before them are already in the ring, the chunk's own K (after RoPE) and V
 * come in k_chunk / v_chunk, not yet in the cache -- a chunk may be longer
 * than the ring.  Query i (at position kv_len - q_len + i) attends keys t <=
 * its position with t > position - window: exactly what
 * pkv_prefill_attention_ragged computes over a linear cache that holds the
 * whole sequence (e4m3 rings: the chunk's keys quantised as
 * pkv_append_rope quantises them).  Then the call commits the chunk: its
 * last R * 16 tokens are written into the ring as pkv_append_rope writes
 * them (no rotation), leaving the ring ready for the next decode step.
 * Three launches on `stream`: staging of each sequence's visible window
 * (ring keys and chunk keys, bf16; e4m3 codes widened exactly) into the
 * workspace, the commit, and the prefill over the staged copy.
 *   k_chunk, v_chunk: bf16 [total_q_tokens][Hkv][D].
 *   block_tables: int32 [num_seqs][max_blocks_per_seq], the first R entries
 *               the ring's blocks.  kv_lens (device) and kv_lens_host: the
 *               lengths after the chunk.  qo_indptr_host and kv_lens_host
 *               are required.
 *   window   : > 0, with every window fitting the ring (PKV_ERR_INVALID_ARG).
 *   workspace: >= pkv_prefill_ring_workspace_size(desc, num_seqs, window,
 *               max q_len) bytes, 256-byte aligned, no initial contents.
 * Other arguments as in pkv_prefill_attention_ragged. */
pkv_status pkv_prefill_ring_commit(const pkv_cache_desc *desc, const void *q, const int32_t *qo_indptr,
                                   const void *k_chunk, const void *v_chunk, void *k_cache, void *v_cache,
                                   const float *k_scale, const float *v_scale, const int32_t *block_tables,
                                   const int32_t *kv_lens, int32_t num_seqs, int32_t total_q_tokens,
                                   const int32_t *qo_indptr_host, const int32_t *kv_lens_host,
                                   float sm_scale, int32_t window, void *out, float *lse_out,
                                   void *workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Host: workspace bytes pkv_prefill_ring_commit needs; 0 for invalid arguments. */
size_t pkv_prefill_ring_workspace_size(const pkv_cache_desc *desc, int32_t num_seqs, int32_t window,
                                       int32_t max_q_len);

/* Host: workspace bytes pkv_prefill_attention_ragged needs: 0 (every path
 * reads bf16 and e4m3 pools directly; kept so that callers may size one). */
size_t pkv_prefill_workspace_size(const pkv_cache_desc *desc, int32_t num_seqs,
                                  int32_t total_q_tokens);

/* ---- a5: merge of partial attention states (FlashAttention-2) -----------
 * For P parts over disjoint key sets: M = max_i lse_i, w_i = exp(lse_i - M),
 *   out = sum_i w_i o_i / sum_i w_i,  lse_out = M + ln sum_i w_i.
 * Parts with lse = -inf are empty (weight 0, their o never read); if all are
 * empty out = 0, lse_out = -inf.
 *   o_parts : fp32 [num_parts][num_rows][num_heads][head_dim].
 *   lse_parts: fp32 [num_parts][num_rows][num_heads].
 *   out     : bf16 [num_rows][num_heads][head_dim].  lse_out: nullable. */
pkv_status pkv_merge_states(const float *o_parts, const float *lse_parts, int32_t num_parts,
                            int32_t num_rows, int32_t num_heads, int32_t head_dim, void *out,
                            float *lse_out, pkv_stream_t stream);

/* ---- f2: cascade (shared-prefix) decode --------------------------------
 * Decode for batches whose sequences share cached prefixes (infer-lab,
 * "Technique" table: RadixAttention prefix caching, and its invariant
 * "prefix-cached == uncached"; llm-infer, "What It Does": prefix caching for
 * prompts that share leading blocks).  Sequences come in groups of
 * consecutive indices; sequence s of group g attends the keys of its group's
 * prefix (prefix_lens[g] tokens through prefix_tables[g]) followed by the
 * keys of its own suffix (suffix_lens[s] tokens through suffix_tables[s]):
 *   o = softmax(sm_scale * q k^T) v over prefix and suffix keys together,
 * the same result as pkv_decode_attention over the concatenated table.  The
 * group's queries attend the prefix in one pass that reads each prefix block
 * once for the whole group; the suffixes go through the split-KV decode;
 * the two (o, lse) states merge as in pkv_merge_states.
 *   q, out    : bf16 [num_seqs][Hq][D].  lse_out: fp32 [num_seqs][Hq], nullable.
 *   group_indptr (device) / group_indptr_host (host): int32 [num_groups+1],
 *               0 = group_indptr[0] <= ... <= group_indptr[num_groups] = num_seqs.
 *   prefix_tables: int32 [num_groups][max_blocks_per_seq]; prefix_lens (device)
 *               and prefix_lens_host: int32 [num_groups], tokens in [0, table capacity].
 *   suffix_tables: int32 [num_seqs][max_blocks_per_seq]; suffix_lens: int32
 *               [num_seqs], each in [1, max_suffix_len] (the new token is in the suffix).
 *   k_scale, v_scale: fp32 [Hkv], e4m3 pools only (else NULL), as in
 *               pkv_decode_attention; every pass reads the codes directly.
 *   window   : <= 0 for full attention; > 0 a sliding window over each
 *               sequence's positions (its query at prefix + suffix_len - 1
 *               sees keys t > that position - window).  A window reaches at
 *               most window - 1 prefix keys, the last ones, and they differ
 *               per sequence: the prefix pass is then the split-KV decode
 *               over the group's prefix table, each sequence from its own
 *               window start.
 *   workspace : >= pkv_cascade_workspace_size(...) bytes, 256-byte aligned,
 *               zero-filled before its first use (it holds the decode tickets).
 * No ring cache (PKV_ERR_UNSUPPORTED). */
pkv_status pkv_cascade_decode(const pkv_cache_desc *desc, const void *q, const void *k_cache,
                              const void *v_cache, const float *k_scale, const float *v_scale,
                              int32_t num_groups, const int32_t *group_indptr,
                              const int32_t *group_indptr_host, const int32_t *prefix_tables,
                              const int32_t *prefix_lens, const int32_t *prefix_lens_host,
                              int32_t num_seqs, const int32_t *suffix_tables,
                              const int32_t *suffix_lens, int32_t max_suffix_len, float sm_scale,
                              int32_t window, void *out, float *lse_out, void *workspace,
                              size_t workspace_bytes, pkv_stream_t stream);

/* Host: workspace bytes pkv_cascade_decode needs for these bounds (planning
 * uses the current device's SM count); 0 for invalid arguments. */
size_t pkv_cascade_workspace_size(const pkv_cache_desc *desc, int32_t num_groups, int32_t num_seqs,
                                  int32_t max_prefix_len, int32_t max_suffix_len, int32_t window);

/* ---- decode with no workspace argument (no counterpart on the pages) ---
 * The same computation as pkv_decode_attention, for callers that cannot
 * allocate device memory at the point of the call -- for example code that
 * runs inside an allocator's own callbacks, under a framework that owns and
 * locks the memory pool, or in a plugin that is handed only the tensors it
 * reads and writes -- and so cannot pass the decode workspace.  Instead of a
 * caller workspace it uses one fixed scratch array of 16 MiB (256-byte
 * aligned) that lives in the library's device memory: every GPU that loads
 * libpkv holds its own copy until the process exits.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - A batch whose split plan needs more than 16 MiB of scratch (see
 *     pkv_decode_workspace_size) is rejected with PKV_ERR_WORKSPACE; pass a
 *     larger chunk_blocks, or use pkv_decode_attention.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents.
 *     A plan of more than four chunks per (sequence, KV head) merges through
 *     tickets kept in the array: such a call first clears them on `stream`
 *     (cudaMemsetAsync, which allocates nothing).  Plans of two to four
 *     chunks merge in shared memory and one-chunk plans need no scratch.
 *     Calls that overlap on the GPU (different streams, or several host
 *     threads) race on the array: serialise them.
 * Arguments are those of pkv_decode_attention without workspace and
 * workspace_bytes. */
pkv_status pkv_decode_attention_static(const pkv_cache_desc *desc, const void *q,
                                       const void *k_cache, const void *v_cache,
                                       const float *k_scale, const float *v_scale,
                                       const int32_t *block_tables, const int32_t *context_lens,
                                       int32_t num_seqs, int32_t max_context_len, float sm_scale,
                                       int32_t window, const float *sinks, int32_t chunk_blocks,
                                       void *out, float *lse_out, pkv_stream_t stream);

/* ---- diagnostics --------------------------------------------------------- */

/* Message for the last non-OK status on this thread ("" if none). */
const char *pkv_last_error(void);

/* Testing only (no counterpart on the pages): make the library's bounded
 * waits give up on purpose, to exercise their failure path without a fault.
 * kernels: bit 0 arms the decode kernel (pkv_decode_attention / _step /
 * _static), bit 1 the tcgen05 prefill kernel; 0 disarms (the default).
 * While armed, every launch of those kernels replaces the first pipeline wait
 * of one warp of its first CTA by a wait on a barrier that nothing arrives
 * on, which gives up after limit_us (1 .. 1000000).  The kernel then drains
 * the copies and MMAs it issued (they all complete), sets
 * PKV_DEVERR_TIMEOUT, writes o = 0 / lse = -inf for the affected state and
 * returns; every merge ticket is left at zero.  Process-wide, not for use
 * in production. */
pkv_status pkv_test_inject_wait_timeout(int32_t kernels, uint32_t limit_us);

/* Host, synchronous: copy the current device's error word (PKV_DEVERR_*
 * bits set by kernels since the last reset) to *flags_out; reset != 0
 * clears it.  Waits for the device to finish preceding work. */
pkv_status pkv_device_errors(uint32_t *flags_out, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
