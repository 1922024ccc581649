// internal.h -- host-side interface between the C ABI layer (api.cu) and the
// kernel translation units.  Launchers return cudaGetLastError() of their
// launch; argument validation happens in api.cu before they are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct AppendArgs {
    void* k_cache;
    void* v_cache;
    const float* k_scale;
    const float* v_scale;
    const int32_t* block_tables;
    const int32_t* token_to_seq;
    const int32_t* positions;
    const void* k_new;
    const void* v_new;
    void* q;  // nullable
    const float* cos_sin;  // nullable
    int32_t num_seqs, num_tokens, hq, hkv, d, mbps, max_pos;
    int64_t num_blocks;
    int32_t fp8;
    int32_t ring;  // > 0: table entry (p / 16) % ring
    uint32_t* err;
};
cudaError_t launch_append_rope(const AppendArgs& a, cudaStream_t stream);

struct GatherArgs {
    const void* cache;
    const int32_t* block_tables;
    const int32_t* lens;
    const int32_t* cu_lens;
    void* out;
    int32_t num_seqs, hkv, row_bytes, mbps;
    int64_t total_tokens, num_blocks;
    uint32_t* err;
};
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);

struct CopyArgs {
    void* k_cache;
    void* v_cache;
    const int32_t* src;
    const int32_t* dst;
    int32_t num_pairs;
    int64_t num_blocks, block_bytes;
    uint32_t* err;
};
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);

// Ring-cache prefill (RustInfer, "Status": Tensor Core prefill over an SWA
// ring cache, followed by a stream-ordered cache commit).  Sequence s has
// q_len = qo_indptr[s+1] - qo_indptr[s] new tokens at positions [kv_len -
// q_len, kv_len); its earlier keys live in a ring of `ring` table entries
// (position p in entry (p / 16) % ring).  Staging copies, per sequence, the
// keys at positions [start, kv_len) that the chunk's window can see --
// start = the block floor of max(0, kv_len - q_len - window + 1) -- into
// staging blocks s * cap .. s * cap + cap - 1 (bf16; e4m3 codes become their
// exact bf16 values, the chunk's own e4m3 keys are quantised first), so the
// prefill runs over a linear table of kv_len - start keys.  The commit then
// writes the chunk's last ring * 16 tokens into the ring.
struct RingStageArgs {
    const void* k_cache;   // the ring pools, bf16 or e4m3
    const void* v_cache;
    const float* k_scale;  // e4m3 only
    const float* v_scale;
    const int32_t* block_tables;  // [num_seqs][mbps], ring entries in the first `ring`
    const int32_t* qo_indptr;
    const int32_t* kv_lens;
    const void* k_chunk;   // bf16 [total_q][hkv][d]: the chunk's K (after RoPE) and V
    const void* v_chunk;
    uint16_t* k_stage;     // bf16 [num_seqs * cap][hkv][16][d]
    uint16_t* v_stage;
    int32_t* stage_tables; // [num_seqs][cap]
    int32_t* stage_lens;   // [num_seqs]: kv_len - start
    void* k_ring_out;      // the pools again, written by the commit
    void* v_ring_out;
    int32_t num_seqs, hkv, d, mbps, ring, window, cap, fp8, total_q;
    int64_t num_blocks;
    uint32_t* err;
};
cudaError_t launch_stage_ring(const RingStageArgs& a, cudaStream_t stream);
cudaError_t launch_commit_ring(const RingStageArgs& a, cudaStream_t stream);

struct MergeArgs {
    const float* o_parts;
    const float* lse_parts;
    void* out;
    float* lse_out;
    int32_t num_parts, num_rows, num_heads, head_dim;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

struct DecodeArgs {
    const void* q;
    void* out;
    float* out_f32;  // non-null: fp32 output (an (o, lse) state to merge) instead of bf16 out
    float* lse_out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const float* k_scale;
    const float* v_scale;
    const float* sinks;   // nullable: fp32 [hq] sink logits
    uint32_t* counters;   // [num_seqs * hkv], zero on entry and exit
    float* part_lse;      // [num_seqs * hkv * max_splits * group]
    float* part_o;        // [num_seqs * hkv * max_splits * group * d]
    uint32_t* err;
    int32_t num_seqs, hq, hkv, group, d, mbps, window, chunk_blocks, max_splits, fp8;
    int32_t max_ctx;  // host bound on context_lens: the split plan covers up to it
    int32_t ring;     // > 0: logical block b is table entry b % ring
    int64_t num_blocks;
    float sm_scale;
    // Fused append (decode step): when k_new is set, every sequence's new
    // token (position context_lens[s] - 1) is written into its cache row by
    // the warp that loads that block, before the load; cos_sin (nullable)
    // rotates it and q.
    const void* k_new;      // bf16 [num_seqs][hkv][d]
    const void* v_new;      // bf16 [num_seqs][hkv][d]
    const float* cos_sin;   // fp32 [max_pos][d/2][2]
    void* k_pool;           // the pools the tensor maps view, written
    void* v_pool;
    // defer_wait != 0: the launch reads nothing the previous kernel in the
    // stream writes (that kernel only waited for its own predecessors), so
    // it starts without the grid-dependency wait and takes it before exiting
    int32_t defer_wait;
    // early_kv != 0: the previous kernel in the stream writes none of the
    // block-table entries, lengths and K/V rows this launch reads (only what
    // it reads through q, k_new, v_new, cos_sin): the lengths, the block ids
    // and the first ring loads are issued before the grid-dependency wait
    int32_t early_kv;
    // test hook: inject_timeout != 0 makes warp 0 of CTA (0, 0, 0) give up
    // its first pipeline wait after inject_limit_us (see common.cuh)
    int32_t inject_timeout;
    uint32_t inject_limit_us;
    // Windowed cascade prefix pass (group_indptr != null): sequence s reads
    // table row and context length g, its group (group_indptr[g] <= s <
    // group_indptr[g + 1]), with visible keys [ctx + group_suffix_lens[s] -
    // window, ctx): the prefix keys its query's window reaches.
    const int32_t* group_indptr;
    const int32_t* group_suffix_lens;
    int32_t num_groups;
};
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream);
// True when a plan of `splits` chunks per (sequence, KV head) merges through
// the workspace tickets (more chunks than one cluster merges).
bool decode_uses_tickets(int splits);

constexpr int kPrefillOrderMax = 256;  // sequences the prefill launch can reorder
struct PrefillArgs {
    const void* q;
    const float* k_scale;  // nullable: per KV head, folded into the logit scale (staged FP8 pools)
    const float* v_scale;  // nullable: per KV head, folded into the output
    void* out;
    float* out_f32;  // non-null: fp32 output (an (o, lse) state to merge) instead of bf16 out
    float* lse_out;
    const int32_t* qo_indptr;
    const int32_t* kv_lens;
    const int32_t* block_tables;
    uint32_t* err;
    int32_t num_seqs, hq, hkv, group, d, mbps, causal, window, max_qtiles, q_tile;
    int32_t total_q;  // rows of q / out
    // tcgen05 kernel: fp8 != 0 reads e4m3 pools (tensor maps of one unswizzled
    // box per (block, head)) and converts each tile to f16 in shared memory
    int32_t fp8;
    int64_t num_blocks;
    float sm_scale;
    // ordered != 0: grid z index i runs sequence seq_order[i], the host's
    // order of decreasing work, so the heaviest CTAs are dispatched first
    int32_t ordered;
    uint16_t seq_order[kPrefillOrderMax];
    // short-query kernel (short_query.cu): blocks per chunk, chunks per
    // (sequence, KV head) (<= kSqMaxSplits; > 1 launches clusters) and m16
    // row tiles per CTA (rows = q_len * group <= 16 * this)
    int32_t sq_chunk, sq_splits, sq_row_tiles;
    // test hook: inject_timeout != 0 makes the MMA warp of CTA (0, 0, 0) of
    // the tcgen05 kernel give up its first K-tile wait after inject_limit_us
    int32_t inject_timeout;
    uint32_t inject_limit_us;
};
constexpr int kSqMaxRowTiles = 4;   // 64 query rows (tokens x heads of a KV group)
constexpr int kSqMaxSplits = 4;     // chunks per (sequence, KV head): one cluster
constexpr int kSqMaxChunk = 512;    // blocks per chunk (a warp's ids: 4 per lane)
// Ragged attention of at most 64 query rows per (sequence, KV head) over bf16
// pools; tensor maps as for decode (one 5-D box per (block, head) tile).
cudaError_t launch_short_query(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream);
// Query tokens per CTA tile for a group size (rows = tokens * group <= 128).
int prefill_tc_q_tile(int group);
// qmap: 3-D tiled view of q [total_q][Hq][D], box {64, G, q_tile}, 128-byte swizzle.
cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t stream);

// Tensor-map box shape used by the attention kernels for a pool:
// innermost box extent in elements, and the swizzle.
struct BoxShape {
    int inner;  // elements per box row
    int boxes;  // boxes per (block, head) tile
    int swizzle128;
};
BoxShape kv_box_shape(int head_dim, int fp8);

}  // namespace pkv
