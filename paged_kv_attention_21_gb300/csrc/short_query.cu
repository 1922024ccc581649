// short_query.cu -- attention of a few query tokens per sequence over the
// paged cache: speculative verify (q_len 2-8 tokens; infer-lab, "Technique"
// table: speculative decoding) and the queries of a group over its shared
// prefix (cascade decode; infer-lab, "Technique" table: prefix caching).
//
// What it computes is the ragged attention of prefill_tc.cu: query token i of
// a sequence with q_len queries and kv_len keys sits at position
// kv_len - q_len + i and sees keys t < kv_len, t <= that position when
// causal, and t > position - window with a window; o = softmax(sm_scale q K^T) V.
//
// Why a second kernel: a 128-row tcgen05 tile holds at most 64 useful rows
// here (q_len x G), so the tensor-core prefill spends its per-tile cost on
// padding and runs near a third of HBM speed.  This kernel is decode-shaped:
// the rows (query token, head of the KV group), at most 64, are cut into
// m16 tiles and a CTA owns one tile of one chunk of the KV range; its 4 warps
// take the chunk's blocks round-robin, each with its own 2-stage TMA ring,
// and combine in shared memory.  The row tiles of a sequence run side by
// side and read the same blocks, mostly from L2.  A KV range is cut into at
// most 4 chunks; 2-4 chunks launch as a thread-block cluster and merge
// through distributed shared memory, so no workspace is needed.
#include "common.cuh"
#include "internal.h"

namespace pkv {

namespace {

constexpr int kSqWarps = 4;
constexpr int kSqThreads = kSqWarps * 32;
constexpr int kSqStages = 2;  // per-warp ring of (K, V) block tiles

template <int D, bool kFp8 = false>
struct SqCfg {
    // one (block, head) tile: bf16 (128-byte swizzled slices) or e4m3 (one
    // unswizzled row of D bytes per token)
    static constexpr int kTileBytes = kBlockSize * D * (kFp8 ? 1 : 2);
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kWarpBytes = kSqStages * kStageBytes;
    static constexpr int kCombStride = D + 8;  // fp32 row stride of the combine buffer
    static constexpr int kCombBytes = kSqWarps * 16 * kCombStride * 4;
    static constexpr int kBodyBytes = kSqWarps * kWarpBytes > kCombBytes ? kSqWarps * kWarpBytes : kCombBytes;
    static constexpr int kSmemBytes = kBodyBytes + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk `chunk` of row r of a 16 x D bf16 tile as the
// 128-byte-swizzled 5-D TMA box writes it (row r's D/64 slices side by side,
// unit u = r D/64 + chunk / 8, chunks swizzled by u % 8).
template <int D>
__device__ __forceinline__ uint32_t sq_off(int r, int chunk) {
    const int u = r * (D / 64) + (chunk >> 3);
    return static_cast<uint32_t>(u * 128 + (((chunk & 7) ^ (u & 7)) << 4));
}

// One CTA = (chunk, KV head and 16-row tile, sequence).  Rows of tile t are
// R = 16 t + r -> query token R / G, head R % G of the KV group.
// kFp8: e4m3 pools, read straight into f16 MMA fragments as the decode
// kernel does (K words of the raw rows with q in the same dim order, V token
// pairs joined by a byte permute, O dims permuted and put back in the
// combine); P is f16 and the scales fold into the logit scale and the output.
template <int D, bool kFp8, bool kCluster>
__global__ void __launch_bounds__(kSqThreads) short_query_kernel(const PrefillArgs a,
                                                                 const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap) {
    using C = SqCfg<D, kFp8>;
    constexpr int KSTEPS = D / 16;
    constexpr int NTILES = D / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bars[kSqWarps][kSqStages];
    __shared__ float s_m[kSqWarps][16];
    __shared__ float s_l[kSqWarps][16];
    __shared__ int s_flag;

    pdl_wait();
    pdl_launch_dependents();
    const int split = blockIdx.x;
    const int kvh = blockIdx.y / a.sq_row_tiles;
    const int tile = blockIdx.y % a.sq_row_tiles;
    const int seq = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;

    const int q0 = a.qo_indptr[seq];
    const int q_len = a.qo_indptr[seq + 1] - q0;
    const int rows = q_len * G;
    if (q_len <= 0 || 16 * tile >= rows) return;  // no rows in this tile
    int kv_len = a.kv_lens[seq];
    const int cap = a.mbps * kBlockSize;
    if (q0 < 0 || q0 + q_len > a.total_q || rows > 16 * a.sq_row_tiles || (a.causal && kv_len < q_len)) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, PKV_DEVERR_POSITION);
        return;
    }
    if (kv_len > cap) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        kv_len = cap;
    }
    const int trows = min(16, rows - 16 * tile);  // valid rows of this tile
    // query i sits at position off + i; the keys any row may see: [klo, kv_len)
    const int off = kv_len - q_len;
    const int klo = (a.window > 0) ? max(0, off - a.window + 1) : 0;
    if (kv_len <= 0 || klo >= kv_len) {  // no visible key: o = 0, lse = -inf
        if (split == 0) {
            for (int i = threadIdx.x; i < trows * D; i += kSqThreads) {
                const int R = 16 * tile + i / D;
                const size_t orow = static_cast<size_t>(q0 + R / G) * a.hq + kvh * G + R % G;
                if (a.out_f32)
                    a.out_f32[orow * D + i % D] = 0.f;
                else
                    static_cast<__nv_bfloat16*>(a.out)[orow * D + i % D] = __float2bfloat16_rn(0.f);
                if (a.lse_out && i % D == 0) a.lse_out[orow] = -INFINITY;
            }
        }
        return;
    }
    const int first_blk = klo / kBlockSize;
    const int last_blk = (kv_len - 1) / kBlockSize;
    int nsplit = (last_blk - first_blk + a.sq_chunk) / a.sq_chunk;
    if (nsplit > a.sq_splits) {  // lengths beyond the host's plan: flagged, never a rank past the cluster
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        nsplit = a.sq_splits;
    }
    if (split >= nsplit) return;
    const int b0 = first_blk + split * a.sq_chunk;
    const int b1 = min(last_blk + 1, b0 + a.sq_chunk);
    const int my_n = (b1 - b0 > warp) ? (b1 - b0 - warp + kSqWarps - 1) / kSqWarps : 0;  // <= 128

    if (threadIdx.x < kSqWarps * kSqStages) mbar_init(&bars[threadIdx.x / kSqStages][threadIdx.x % kSqStages], 1);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        s_flag = 0;
    }
    fence_barrier_init();
    __syncthreads();

    // this warp's blocks b0 + warp + 4 k; lane l holds the ids of k = l, l + 32, l + 64, l + 96
    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.mbps;
    int ids[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int kk = lane + 32 * j;
        int id = 0;
        if (kk < my_n) {
            id = bt[b0 + warp + kSqWarps * kk];
            if (id < 0 || id >= a.num_blocks) {
                flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                id = 0;  // read a valid block; the output is flagged invalid
            }
        }
        ids[j] = id;
    }
    auto block_id = [&](int kk) {  // warp-uniform kk < 128
        const int j = kk >> 5;
        const int v = j == 0 ? ids[0] : j == 1 ? ids[1] : j == 2 ? ids[2] : ids[3];
        return __shfl_sync(0xFFFFFFFFu, v, kk & 31);
    };
    uint8_t* wbase = smem + warp * C::kWarpBytes;
#pragma unroll
    for (int kk = 0; kk < kSqStages; ++kk) {
        const int pb = block_id(kk);
        if (lane == 0 && kk < my_n) {
            uint8_t* dst = wbase + kk * C::kStageBytes;
            mbar_arrive_expect_tx(&bars[warp][kk], C::kStageBytes);
            if constexpr (kFp8) {
                tma_load_4d(dst, &kmap, &bars[warp][kk], 0, 0, kvh, pb);
                tma_load_4d(dst + C::kTileBytes, &vmap, &bars[warp][kk], 0, 0, kvh, pb);
            } else {
                tma_load_5d(dst, &kmap, &bars[warp][kk], 0, 0, 0, kvh, pb);
                tma_load_5d(dst + C::kTileBytes, &vmap, &bars[warp][kk], 0, 0, 0, kvh, pb);
            }
        }
    }

    // rows of the tile: lane rows g0 and g0 + 8
    const int g0 = lane >> 2;
    const int tig = lane & 3;
    int hi_r[2], lo_r[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = g0 + 8 * h;
        const int pos = off + (16 * tile + r) / G;  // the window is relative to the query's position
        hi_r[h] = r < trows ? (a.causal ? pos : kv_len - 1) : -1;  // padding rows see no key
        lo_r[h] = a.window > 0 ? max(0, pos - a.window + 1) : 0;
    }
    uint32_t qa[KSTEPS][4];
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const int r = g0 + ((part & 1) ? 8 : 0);
            // e4m3: k-step kk of lane (g, tig) covers dims tig D/4 + 4 kk + {0..3},
            // the order its K words come in (the dot product is a sum over dims)
            const int col = kFp8 ? tig * (D / 4) + 4 * kk + ((part & 2) ? 2 : 0)
                                 : kk * 16 + 2 * tig + ((part & 2) ? 8 : 0);
            uint32_t v = 0;
            if (r < trows) {
                const int R = 16 * tile + r;
                const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                            (static_cast<size_t>(q0 + R / G) * a.hq + kvh * G + R % G) * D;
                v = *reinterpret_cast<const uint32_t*>(qrow + col);
                if constexpr (kFp8) v = pack2<true>(bf16_lo(v), bf16_hi(v));
            }
            qa[kk][part] = v;
        }
    }
    const float scale_log2 = a.sm_scale * 1.4426950408889634f * (a.k_scale ? a.k_scale[kvh] : 1.f);

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[NTILES][4];
#pragma unroll
    for (int nt = 0; nt < NTILES; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    bool failed = false;
    int k = 0;
    for (; k < my_n; ++k) {
        const int st = k % kSqStages;
        const uint32_t ph = (k / kSqStages) & 1;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars[warp][st], ph))) {
            failed = true;
            break;
        }
        const uint32_t kaddr = smem_u32(wbase + st * C::kStageBytes);
        const uint32_t vaddr = kaddr + C::kTileBytes;
        const int tok_base = (b0 + warp + k * kSqWarps) * kBlockSize;

        // ---- S = Q . K^T  (16 rows x 16 tokens)
        float sacc[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
        if constexpr (kFp8) {
            // rows g (tokens 0-7) and g + 8 (tokens 8-15), bytes [tig D/4, (tig+1) D/4)
            const uint8_t* ktile = wbase + st * C::kStageBytes;
            uint32_t kw[2][D / 16];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int q4 = 0; q4 < D / 64; ++q4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(ktile + (g0 + 8 * n) * D + tig * (D / 4) + 16 * q4);
                    kw[n][4 * q4] = v.x;
                    kw[n][4 * q4 + 1] = v.y;
                    kw[n][4 * q4 + 2] = v.z;
                    kw[n][4 * q4 + 3] = v.w;
                }
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t b0, b1, b2, b3;
                e4m3x4_to_f16x4(kw[0][kk], b0, b1);
                e4m3x4_to_f16x4(kw[1][kk], b2, b3);
                mma_16816<true>(sacc[0], qa[kk], b0, b1);
                mma_16816<true>(sacc[1], qa[kk], b2, b3);
            }
        } else {
            const int tok = (lane & 7) + ((lane >> 4) << 3);
            const int csel = (lane >> 3) & 1;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t b00, b01, b10, b11;
                ldmatrix_x4(b00, b01, b10, b11, kaddr + sq_off<D>(tok, 2 * kk + csel));
                mma_16816<false>(sacc[0], qa[kk], b00, b01);
                mma_16816<false>(sacc[1], qa[kk], b10, b11);
            }
        }
        // ---- per-row mask + online softmax (exp2 domain)
        float x[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                const int t = tok_base + n * 8 + 2 * tig + (e & 1);
                x[n][e] = (t < lo_r[h] || t > hi_r[h]) ? -INFINITY : sacc[n][e] * scale_log2;
            }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
        const float mn0 = fmaxf(m_run[0], mx0);
        const float mn1 = fmaxf(m_run[1], mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m_run[0] - mu0);
        const float al1 = fast_exp2(m_run[1] - mu1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        float p[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            p[n][0] = fast_exp2(x[n][0] - mu0);
            p[n][1] = fast_exp2(x[n][1] - mu0);
            p[n][2] = fast_exp2(x[n][2] - mu1);
            p[n][3] = fast_exp2(x[n][3] - mu1);
        }
        l_run[0] = l_run[0] * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        l_run[1] = l_run[1] * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
        if (__any_sync(0xFFFFFFFFu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int nt = 0; nt < NTILES; ++nt) {
                o[nt][0] *= al0;
                o[nt][1] *= al0;
                o[nt][2] *= al1;
                o[nt][3] *= al1;
            }
        }
        uint32_t pa[4];
        pa[0] = pack2<kFp8>(p[0][0], p[0][1]);
        pa[1] = pack2<kFp8>(p[0][2], p[0][3]);
        pa[2] = pack2<kFp8>(p[1][0], p[1][1]);
        pa[3] = pack2<kFp8>(p[1][2], p[1][3]);
        // ---- O += P . V, V rows outside [klo, kv_len) zeroed (0 * NaN never
        // reaches the MMA)
        uint32_t keep_lo = 0xFFFFFFFFu, keep_hi = 0xFFFFFFFFu;
        if (tok_base < klo || tok_base + kBlockSize > kv_len) {
            const int t0 = tok_base + 2 * tig;
            const bool v0 = t0 >= klo && t0 < kv_len, v1 = t0 + 1 >= klo && t0 + 1 < kv_len;
            const bool v8 = t0 + 8 >= klo && t0 + 8 < kv_len, v9 = t0 + 9 >= klo && t0 + 9 < kv_len;
            keep_lo = (v0 ? 0x0000FFFFu : 0u) | (v1 ? 0xFFFF0000u : 0u);
            keep_hi = (v8 ? 0x0000FFFFu : 0u) | (v9 ? 0xFFFF0000u : 0u);
        }
        if constexpr (kFp8) {
            // lane (g, tig) takes dims [g D/8, (g+1) D/8) of V rows 2 tig, 2 tig + 1
            // (b0) and 2 tig + 8, 2 tig + 9 (b1); n-tile nt's column is dim g D/8 + nt
            constexpr int W = D / 32;  // 32-bit words of a lane's slice of one row
            const uint8_t* vb = wbase + st * C::kStageBytes + C::kTileBytes + g0 * (D / 8);
            uint32_t r0[W], r1[W], r8[W], r9[W];
            auto row_words = [&](int row, uint32_t (&w)[W]) {
                if constexpr (W == 2) {
                    const uint2 t = *reinterpret_cast<const uint2*>(vb + row * D);
                    w[0] = t.x;
                    w[1] = t.y;
                } else {
                    const uint4 t = *reinterpret_cast<const uint4*>(vb + row * D);
                    w[0] = t.x;
                    w[1] = t.y;
                    w[2] = t.z;
                    w[3] = t.w;
                }
            };
            row_words(2 * tig, r0);
            row_words(2 * tig + 1, r1);
            row_words(2 * tig + 8, r8);
            row_words(2 * tig + 9, r9);
#pragma unroll
            for (int nt = 0; nt < NTILES; nt += 2) {
                // bytes s, s+1 of word nt/4 from both rows of a pair: (a_s, b_s, a_s+1, b_s+1)
                const uint32_t sel = (nt % 4 == 0) ? 0x5140u : 0x7362u;
                uint32_t plo, phi;
                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(plo) : "r"(r0[nt / 4]), "r"(r1[nt / 4]), "r"(sel));
                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(phi) : "r"(r8[nt / 4]), "r"(r9[nt / 4]), "r"(sel));
                uint32_t b0a, b0b, b1a, b1b;
                e4m3x4_to_f16x4(plo, b0a, b0b);
                e4m3x4_to_f16x4(phi, b1a, b1b);
                b0a &= keep_lo;
                b0b &= keep_lo;
                b1a &= keep_hi;
                b1b &= keep_hi;
                mma_16816<true>(o[nt], pa, b0a, b1a);
                mma_16816<true>(o[nt + 1], pa, b0b, b1b);
            }
        } else {
            const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
            const int csel = lane >> 4;
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(v0, v1, v2, v3, vaddr + sq_off<D>(tok, 2 * j + csel));
                v0 &= keep_lo;
                v2 &= keep_lo;
                v1 &= keep_hi;
                v3 &= keep_hi;
                mma_16816<false>(o[2 * j], pa, v0, v1);
                mma_16816<false>(o[2 * j + 1], pa, v2, v3);
            }
        }
        __syncwarp();
        // refill this stage with the block NSTAGE ahead (the stage was only
        // read, and the reads' values are consumed: no proxy fence needed)
        const int kn = k + kSqStages;
        const int pb = block_id(kn & 127);
        if (lane == 0 && kn < my_n) {
            uint8_t* dst = wbase + st * C::kStageBytes;
            mbar_arrive_expect_tx(&bars[warp][st], C::kStageBytes);
            if constexpr (kFp8) {
                tma_load_4d(dst, &kmap, &bars[warp][st], 0, 0, kvh, pb);
                tma_load_4d(dst + C::kTileBytes, &vmap, &bars[warp][st], 0, 0, kvh, pb);
            } else {
                tma_load_5d(dst, &kmap, &bars[warp][st], 0, 0, 0, kvh, pb);
                tma_load_5d(dst + C::kTileBytes, &vmap, &bars[warp][st], 0, 0, 0, kvh, pb);
            }
        }
    }
    if (failed) {
        // drain the loads still in flight -- the stage that gave up and the
        // ones after it (bounded) -- so that no copy lands after exit, then report
        for (int kk = k; kk < min(my_n, k + kSqStages); ++kk)
            (void)mbar_wait(&bars[warp][kk % kSqStages], (kk / kSqStages) & 1);
        if (lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            atomicOr(&s_flag, 1);
        }
    }

    // ---- combine the 4 warps of the CTA
    l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], 1);
    l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], 2);
    l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], 1);
    l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], 2);
    __syncthreads();  // every warp is done with its stage buffers
    float* comb = reinterpret_cast<float*>(smem);
    {
        float* cw = comb + warp * 16 * C::kCombStride;
#pragma unroll
        for (int nt = 0; nt < NTILES; ++nt) {
            if constexpr (kFp8) {  // dims 2 tig D/8 + nt and (2 tig + 1) D/8 + nt
                const int c0 = 2 * tig * (D / 8) + nt;
                const int c1 = c0 + D / 8;
                cw[g0 * C::kCombStride + c0] = o[nt][0];
                cw[g0 * C::kCombStride + c1] = o[nt][1];
                cw[(g0 + 8) * C::kCombStride + c0] = o[nt][2];
                cw[(g0 + 8) * C::kCombStride + c1] = o[nt][3];
            } else {
                const int col = nt * 8 + 2 * tig;
                *reinterpret_cast<float2*>(cw + g0 * C::kCombStride + col) = make_float2(o[nt][0], o[nt][1]);
                *reinterpret_cast<float2*>(cw + (g0 + 8) * C::kCombStride + col) =
                    make_float2(o[nt][2], o[nt][3]);
            }
        }
        if (tig == 0) {
            s_m[warp][g0] = m_run[0];
            s_m[warp][g0 + 8] = m_run[1];
            s_l[warp][g0] = l_run[0];
            s_l[warp][g0 + 8] = l_run[1];
        }
    }
    __syncthreads();
    const bool cta_failed = s_flag != 0;
    // per row, once: the warps' weights 2^(m_w - M) / L (v_scale folded in)
    // replace s_m, and the row's lse goes to s_l[0]
    if (threadIdx.x < 16) {
        const int r = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSqWarps; ++w) M = fmaxf(M, s_m[w][r]);
        float f[kSqWarps];
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kSqWarps; ++w) {
            f[w] = s_m[w][r] == -INFINITY ? 0.f : fast_exp2(s_m[w][r] - M);
            L += f[w] * s_l[w][r];
        }
        // a failed chunk contributes nothing: weight 0, lse = -inf
        const float inv = L > 0.f && !cta_failed ? (a.v_scale ? a.v_scale[kvh] : 1.f) / L : 0.f;
        const float lse = L > 0.f && !cta_failed ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
#pragma unroll
        for (int w = 0; w < kSqWarps; ++w) s_m[w][r] = f[w] * inv;
        s_l[0][r] = lse;
    }
    __syncthreads();
    {
        for (int idx = threadIdx.x; idx < trows * D; idx += kSqThreads) {
            const int r = idx / D;
            const int d = idx % D;
            float ov = 0.f;
            if (!cta_failed) {
#pragma unroll
                for (int w = 0; w < kSqWarps; ++w) ov += s_m[w][r] * comb[(w * 16 + r) * C::kCombStride + d];
            }
            if (nsplit == 1) {
                const int R = 16 * tile + r;
                const size_t orow = static_cast<size_t>(q0 + R / G) * a.hq + kvh * G + R % G;
                if (a.out_f32)
                    a.out_f32[orow * D + d] = ov;
                else
                    static_cast<__nv_bfloat16*>(a.out)[orow * D + d] = __float2bfloat16_rn(ov);
                if (a.lse_out && d == 0) a.lse_out[orow] = s_l[0][r];
            } else {
                comb[r * C::kCombStride + d] = ov;  // this chunk's state, in place of warp 0's rows
            }
        }
    }
    if constexpr (kCluster) {
        if (nsplit == 1) return;
        // ---- cluster merge: chunk c holds o_c (warp 0's rows of comb) and lse_c (s_l[0])
        cluster_sync();
        float* wts = comb + 16 * C::kCombStride;  // warp 1's slice, free now: [chunk][16]
        float* rowM = wts + kSqMaxSplits * 16;
        float* rowW = rowM + 16;
        if (threadIdx.x < 16) {
            const int r = threadIdx.x;
            float l[kSqMaxSplits];
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kSqMaxSplits; ++c) {
                l[c] = c < nsplit ? ld_cluster_f32(cluster_map(smem_u32(&s_l[0][r]), c)) : -INFINITY;
                M = fmaxf(M, l[c]);
            }
            float W = 0.f;
#pragma unroll
            for (int c = 0; c < kSqMaxSplits; ++c) {
                const float wv = l[c] == -INFINITY ? 0.f : __expf(l[c] - M);
                wts[c * 16 + r] = wv;
                W += wv;
            }
            rowM[r] = M;
            rowW[r] = W;
        }
        __syncthreads();
        constexpr int kSlotsPerRow = D / 4;
        const int total = trows * kSlotsPerRow;
        const int s_lo = split * total / nsplit;
        const int s_hi = (split + 1) * total / nsplit;
        for (int slot = s_lo + threadIdx.x; slot < s_hi; slot += kSqThreads) {
            const int r = slot / kSlotsPerRow;
            const int c4 = slot % kSlotsPerRow;
            const uint32_t local = smem_u32(comb + r * C::kCombStride + c4 * 4);
            float4 v[kSqMaxSplits];
#pragma unroll
            for (int c = 0; c < kSqMaxSplits; ++c)
                if (c < nsplit) v[c] = ld_cluster_f32x4(cluster_map(local, c));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kSqMaxSplits; ++c) {
                const float w = wts[c * 16 + r];
                if (c < nsplit && w != 0.f) {
                    acc.x += w * v[c].x;
                    acc.y += w * v[c].y;
                    acc.z += w * v[c].z;
                    acc.w += w * v[c].w;
                }
            }
            const float W = rowW[r];
            const float inv = W > 0.f ? 1.f / W : 0.f;
            const int R = 16 * tile + r;
            const size_t orow = static_cast<size_t>(q0 + R / G) * a.hq + kvh * G + R % G;
            if (a.out_f32) {
                *reinterpret_cast<float4*>(a.out_f32 + orow * D + c4 * 4) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            } else {
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * D + c4 * 4) =
                    make_uint2(pack2<false>(acc.x * inv, acc.y * inv), pack2<false>(acc.z * inv, acc.w * inv));
            }
            if (a.lse_out && c4 == 0) a.lse_out[orow] = W > 0.f ? rowM[r] + __logf(W) : -INFINITY;
        }
        cluster_sync();  // no chunk exits while a peer may still read its shared memory
    }
}

template <int D, bool kFp8>
cudaError_t launch_sq_d(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        cudaStream_t stream) {
    using C = SqCfg<D, kFp8>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert((kSqMaxSplits + 2) * 16 <= 16 * C::kCombStride, "cluster merge scratch");
    const bool cluster = a.sq_splits > 1;
    auto kern = cluster ? short_query_kernel<D, kFp8, true> : short_query_kernel<D, kFp8, false>;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[cluster][dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[cluster][dev] = true;
    }
    dim3 grid(a.sq_splits, a.hkv * a.sq_row_tiles, a.num_seqs);
    return launch_pdl_cluster(kern, grid, dim3(kSqThreads), C::kSmemBytes, stream,
                              cluster ? static_cast<unsigned>(a.sq_splits) : 1u, a, kmap, vmap);
}

}  // namespace

cudaError_t launch_short_query(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream) {
    if (a.fp8)
        return a.d == 64 ? launch_sq_d<64, true>(a, kmap, vmap, stream)
                         : launch_sq_d<128, true>(a, kmap, vmap, stream);
    return a.d == 64 ? launch_sq_d<64, false>(a, kmap, vmap, stream)
                     : launch_sq_d<128, false>(a, kmap, vmap, stream);
}

}  // namespace pkv
