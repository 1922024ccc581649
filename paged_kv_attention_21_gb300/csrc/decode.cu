// decode.cu -- split-KV GQA decode attention over the paged cache.
//
// What it computes (FlashAttention-2 work partitioning, cited under
// llm-infer "References"; the paged cache of infer-lab's "Technique" table):
// for sequence s, KV head kvh and each of its G query heads,
//     o = softmax(sm_scale * q K^T) V     over the visible keys,
// where K/V rows are gathered block by block through the block table.
//
// Work decomposition.  The visible blocks of every (sequence, KV head) are
// cut into chunks of `chunk_blocks` blocks (the planner in api.cu); one CTA
// owns one chunk.  Its 4 warps take the chunk's blocks round-robin, each
// warp running its own NSTAGE-deep pipeline of TMA bulk-tensor loads
// (K tile + V tile of one block, 16 rows x D) completed on a per-stage
// mbarrier.  A warp computes, per block,
//     S[16 x 16] = Q[16 x D] . K^T     (mma.sync m16n8k16; rows = the G query
//                                       heads of the group, padded to 16)
//     online softmax on S (running max / sum per row, exp2 domain)
//     O[16 x D] += P[16 x 16] . V
// so ONE read of each K/V block serves the whole GQA group.  At the end the
// 4 warps combine in shared memory; a chunk that is its sequence's only one
// writes bf16 output.  Otherwise the chunks' fp32 (o_i, lse_i) states merge
//     M = max lse_i, w_i = exp(lse_i - M), o = sum w_i o_i / sum w_i
// in the same launch, one of two ways:
//   * plans of 2..4 chunks launch every (sequence, KV head) as a thread-block
//     cluster: each chunk keeps its state in shared memory, and after a
//     cluster barrier every chunk merges a slice of the output by reading its
//     peers' states through distributed shared memory -- no global round
//     trip, no fence;
//   * larger plans write the states to the workspace and take a ticket; the
//     last chunk to arrive merges and resets the ticket.
//
// Decode step (fused append): with k_new set, the warp that loads a
// sequence's last block first writes the new token's K (RoPE) and V rows into
// it, and every CTA rotates its q rows, so append and attention are one launch.
//
// e4m3 pools: the TMA loads fp8 bytes, each warp converts the tile to f16
// (exact) in shared memory and runs the f16 MMA; k_scale folds into the
// logit scale and v_scale into the output.
//
// Roofline: HBM.  Per (block, KV head) the kernel reads 2*16*D*elem bytes
// and does 4*16*D*G flops, G flop/byte for bf16 -- far below the tensor
// pipe's ridge, so the design goal is bytes in flight, not MMA rate.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;  // warps of a CTA (a 2-warp variant serves one-chunk window plans)
// Plans of 2..4 chunks per sequence merge inside a cluster (larger clusters
// measured slower than the ticket merge: co-scheduling them leaves slots idle).
constexpr int kMaxClusterSplits = 4;

template <int D, bool kFp8, int kW = kWarps>
struct DecodeCfg {
    // bf16 tiles: 2 stages per warp keep ~3 CTAs (12 warps) resident per SM,
    // which measured faster than 3 stages at 2 CTAs; e4m3 tiles are small.
    // The 2-warp variant runs windows of at most 9 blocks: with e4m3 tiles a
    // warp's whole share (5 blocks) is in flight after one round of loads.
    static constexpr int kStages = kFp8 ? (kW < kWarps ? 5 : 3) : 2;
    // block-id registers per lane: a warp holds ids for 32 kIdRegs blocks, so
    // a CTA takes chunks of up to 32 kIdRegs kW blocks: 256 with 4 warps on
    // bf16 pools, 128 on e4m3 pools (whose issue-bound loop measured 0.7 %
    // slower with the second register's select)
    static constexpr int kIdRegs = (kW < kWarps || kFp8) ? 1 : 2;
    static constexpr int kElem = kFp8 ? 1 : 2;
    static constexpr int kTileBytes = kBlockSize * D * kElem;  // one block of one head
    static constexpr int kStageBytes = 2 * kTileBytes;         // K + V
    // bf16: one 5-D box per tile (16 rows x D/64 swizzled 128-byte slices);
    // fp8: one unswizzled 4-D box of 16 rows x D bytes
    static constexpr int kConvBytes = kFp8 ? kBlockSize * D * 2 : 0;  // q rows staged once (e4m3)
    static constexpr int kWarpBytes = kStages * kStageBytes + kConvBytes;
    static constexpr int kCombStride = D + 8;  // fp32 row stride of the combine buffer
    static constexpr int kCombBytes = kW * 16 * kCombStride * 4;
    static constexpr int kBodyBytes = kW * kWarpBytes > kCombBytes ? kW * kWarpBytes
                                                                       : kCombBytes;
    static constexpr int kSmemBytes = kBodyBytes + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk `chunk` (0 .. D/8 - 1) of row r in a 16 x D
// 16-bit tile as it sits in shared memory: row r's D/64 slices of 128 bytes
// are side by side (unit u = r D/64 + chunk / 8), and each unit's chunks are
// swizzled by u % 8 -- the layout the 128-byte-swizzled 5-D TMA box writes
// on a 1024-byte aligned tile.  Eight rows at one chunk fall in at most two
// bank groups' worth of conflicts (D = 128) or none (D = 64).
template <int D>
__device__ __forceinline__ uint32_t kv_off(int r, int chunk) {
    const int u = r * (D / 64) + (chunk >> 3);
    return static_cast<uint32_t>(u * 128 + (((chunk & 7) ^ (u & 7)) << 4));
}

// One (block, head) tile of K or V into shared memory.
template <bool kFp8>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int kvh,
                                          int block) {
    if constexpr (kFp8)
        tma_load_4d(dst, map, bar, 0, 0, kvh, block);
    else
        tma_load_5d(dst, map, bar, 0, 0, 0, kvh, block);
}

// Fused append: one warp writes sequence seq's new token (position p) for KV
// head kvh into row p % 16 of physical block blk -- K rotated (RoPE, when
// cos_sin is set) and rounded to bf16 or quantised to e4m3, V copied or
// quantised -- with the same arithmetic as the standalone append kernel, then
// fences the writes against the TMA reads of that block that follow.
// Lane l owns the rotation pairs (j, j + D/2) for j in [l PPL, (l+1) PPL).
template <int D, bool kFp8>
__device__ __forceinline__ void append_new_token(const DecodeArgs& a, int seq, int kvh, int blk, int p,
                                                 int lane) {
    constexpr int HALF = D / 2;
    constexpr int PPL = HALF / 32;
    const int j0 = lane * PPL;
    const size_t src = (static_cast<size_t>(seq) * a.hkv + kvh) * D;
    const size_t dst = ((static_cast<size_t>(blk) * a.hkv + kvh) * kBlockSize + p % kBlockSize) * D;
    const __nv_bfloat16* kx = static_cast<const __nv_bfloat16*>(a.k_new) + src;
    const __nv_bfloat16* vx = static_cast<const __nv_bfloat16*>(a.v_new) + src;
    float lo[PPL], hi[PPL];
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const float av = __bfloat162float(kx[j0 + k]);
        const float bv = __bfloat162float(kx[HALF + j0 + k]);
        if (a.cos_sin) {
            const float c = a.cos_sin[(static_cast<size_t>(p) * HALF + j0 + k) * 2];
            const float sn = a.cos_sin[(static_cast<size_t>(p) * HALF + j0 + k) * 2 + 1];
            lo[k] = __fsub_rn(__fmul_rn(av, c), __fmul_rn(bv, sn));
            hi[k] = __fadd_rn(__fmul_rn(bv, c), __fmul_rn(av, sn));
        } else {
            lo[k] = av;
            hi[k] = bv;
        }
    }
    if constexpr (!kFp8) {
        __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(a.k_pool) + dst;
        __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(a.v_pool) + dst;
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            kc[j0 + k] = __float2bfloat16_rn(lo[k]);
            kc[HALF + j0 + k] = __float2bfloat16_rn(hi[k]);
            vc[j0 + k] = vx[j0 + k];
            vc[HALF + j0 + k] = vx[HALF + j0 + k];
        }
    } else {
        uint8_t* kc = static_cast<uint8_t*>(a.k_pool) + dst;
        uint8_t* vc = static_cast<uint8_t*>(a.v_pool) + dst;
        const float ks = a.k_scale[kvh];
        const float vs = a.v_scale[kvh];
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            kc[j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(lo[k], ks), __NV_SATFINITE, __NV_E4M3);
            kc[HALF + j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(hi[k], ks), __NV_SATFINITE, __NV_E4M3);
            vc[j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(__bfloat162float(vx[j0 + k]), vs), __NV_SATFINITE,
                                               __NV_E4M3);
            vc[HALF + j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(__bfloat162float(vx[HALF + j0 + k]), vs),
                                                      __NV_SATFINITE, __NV_E4M3);
        }
    }
    fence_proxy_async_global();
    __syncwarp();
}

// Q fragments (A operand) of sequence seq's group kvh: rows = the G query
// heads, zero-padded to 16.  rot_pos >= 0 also loads the (cos, sin) pairs
// of that position that rotate_q applies; the loads are only issued here, so
// a caller can overlap them with other work before rotating.
template <int D>
__device__ __forceinline__ void load_q_raw(const DecodeArgs& a, int seq, int kvh, int rot_pos, int lane,
                                           uint32_t (&qa)[D / 16][4], float4 (&cs)[D / 32][2]) {
    constexpr int KSTEPS = D / 16;
    const int G = a.group;
    const int g0 = lane >> 2;
    const int tig = lane & 3;
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q) +
                              (static_cast<size_t>(seq) * a.hq + kvh * G) * D;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const int row = g0 + ((part & 1) ? 8 : 0);
            const int col = kk * 16 + 2 * tig + ((part & 2) ? 8 : 0);
            uint32_t v = 0;
            if (row < G) v = *reinterpret_cast<const uint32_t*>(qb + row * D + col);
            qa[kk][part] = v;
        }
    }
    if (rot_pos >= 0) {
        // column c of k-step kk pairs with column c + D/2 (k-step kk + KSTEPS/2);
        // a lane's columns are kk 16 + 2 tig (+ 8), each with its neighbour c + 1
        const float* t = a.cos_sin + static_cast<size_t>(rot_pos) * (D / 2) * 2;
#pragma unroll
        for (int kk = 0; kk < KSTEPS / 2; ++kk)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                cs[kk][h] = *reinterpret_cast<const float4*>(t + (kk * 16 + 2 * tig + 8 * h) * 2);
    }
}

// RoPE on the Q fragments with the (cos, sin) pairs load_q_raw fetched,
// rounded to bf16 as the standalone append rounds q: columns c, c + 1 sit in
// one register, and their partners c + D/2, c + D/2 + 1 in k-step kk + D/32.
template <int D>
__device__ __forceinline__ void rotate_q(uint32_t (&qa)[D / 16][4], const float4 (&cs)[D / 32][2]) {
    constexpr int KSTEPS = D / 16;
#pragma unroll
    for (int kk = 0; kk < KSTEPS / 2; ++kk) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const float4 t = cs[kk][(part & 2) ? 1 : 0];  // c, s of col, col + 1
            const uint32_t va = qa[kk][part];
            const uint32_t vb = qa[kk + KSTEPS / 2][part];
            const float a0 = bf16_lo(va), a1 = bf16_hi(va);
            const float b0v = bf16_lo(vb), b1v = bf16_hi(vb);
            const float lo0 = __fsub_rn(__fmul_rn(a0, t.x), __fmul_rn(b0v, t.y));
            const float hi0 = __fadd_rn(__fmul_rn(b0v, t.x), __fmul_rn(a0, t.y));
            const float lo1 = __fsub_rn(__fmul_rn(a1, t.z), __fmul_rn(b1v, t.w));
            const float hi1 = __fadd_rn(__fmul_rn(b1v, t.z), __fmul_rn(a1, t.w));
            qa[kk][part] = pack2<false>(lo0, lo1);
            qa[kk + KSTEPS / 2][part] = pack2<false>(hi0, hi1);
        }
    }
}

template <int D>
__device__ __forceinline__ void load_q(const DecodeArgs& a, int seq, int kvh, int rot_pos, int lane,
                                       uint32_t (&qa)[D / 16][4]) {
    float4 cs[D / 32][2];
    load_q_raw<D>(a, seq, kvh, rot_pos, lane, qa, cs);
    if (rot_pos >= 0) rotate_q<D>(qa, cs);
}

// log2 of the largest factor a stale running max may leave in p
constexpr float kLazyRescale = 8.0f;

// One block of K and V (16 tokens of one KV head, in shared memory) into a
// warp's running state:
//     S[16 x 16] = Q . K^T              (rows: the group's query heads, padded)
//     online softmax of S over the keys in [lo, ctx), exp2 domain
//     O[16 x D] += P . V
// tok_base is the block's first token position.  Rows g0 + 8 take part only
// when kHi (a group of more than 8 heads); otherwise they are padding and
// cost no softmax work.
template <int D, bool kFp8, bool kHi>
__device__ __forceinline__ void attend_block(const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4],
                                             float (&m_run)[2], float (&l_run)[2], const uint8_t* ktile,
                                             const uint8_t* vtile, int lane, int tok_base, int lo, int ctx,
                                             float scale_log2) {
    constexpr int kRowVals = kHi ? 4 : 2;  // accumulator values of real rows per n-tile
    constexpr int KSTEPS = D / 16;
    constexpr int NTILES = D / 8;
    const int g0 = lane >> 2;
    const int tig = lane & 3;
    const uint32_t kaddr = smem_u32(ktile);
    const uint32_t vaddr = smem_u32(vtile);

    // ---- S = Q . K^T  (16 heads x 16 tokens)
    float sacc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
    if constexpr (kFp8) {
        // rows g (tokens 0-7 tile) and g + 8 (tokens 8-15 tile), bytes
        // [tig D/4, (tig+1) D/4): word kk -> k-step kk's two f16 pairs
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
            const int chunk = 2 * kk + csel;
            uint32_t b00, b01, b10, b11;
            ldmatrix_x4(b00, b01, b10, b11, kaddr + kv_off<D>(tok, chunk));
            mma_16816<kFp8>(sacc[0], qa[kk], b00, b01);
            mma_16816<kFp8>(sacc[1], qa[kk], b10, b11);
        }
    }
    (void)kaddr;

    // ---- mask + online softmax (exp2 domain)
    const bool edge = tok_base < lo || tok_base + kBlockSize > ctx;
    float x[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[n][e] = e < kRowVals ? sacc[n][e] * scale_log2 : -INFINITY;
    if (edge) {  // the block straddles lo or ctx: token t is visible iff t - lo < ctx - lo (unsigned)
        const int base = tok_base + 2 * tig - lo;
        const uint32_t cnt = static_cast<uint32_t>(ctx - lo);
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < kRowVals; ++e)
                if (static_cast<uint32_t>(base + n * 8 + (e & 1)) >= cnt) x[n][e] = -INFINITY;
    }
    float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
    // Lazy rescale: a row keeps its running max m (p = 2^(x - m) <= 2^8)
    // until a block's max exceeds it by more than 2^8; only then are l and O
    // rescaled.  The final state (m, l, O) is exact for any such m.
    const bool grow0 = mx0 > m_run[0] + kLazyRescale;   // -inf + 8 = -inf: a first finite max grows
    const float mn0 = grow0 ? mx0 : m_run[0];
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float al0 = grow0 ? fast_exp2(m_run[0] - mu0) : 1.f;
    m_run[0] = mn0;
    float p[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        p[n][0] = fast_exp2(x[n][0] - mu0);
        p[n][1] = fast_exp2(x[n][1] - mu0);
        p[n][2] = p[n][3] = 0.f;
    }
    l_run[0] = l_run[0] * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    float al1 = 1.f;
    if constexpr (kHi) {  // rows 8-15 are query heads only when the group has more than 8
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
        const bool grow1 = mx1 > m_run[1] + kLazyRescale;
        const float mn1 = grow1 ? mx1 : m_run[1];
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        al1 = grow1 ? fast_exp2(m_run[1] - mu1) : 1.f;
        m_run[1] = mn1;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            p[n][2] = fast_exp2(x[n][2] - mu1);
            p[n][3] = fast_exp2(x[n][3] - mu1);
        }
        l_run[1] = l_run[1] * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
    }
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

    // ---- O += P . V   (V rows outside the visible range are zeroed so that
    // a NaN in an unused slot never meets a zero weight inside the MMA; with
    // e4m3 tiles a block whose rows are all visible skips the masking)
    uint32_t keep_lo = 0xFFFFFFFFu, keep_hi = 0xFFFFFFFFu;
    if (edge) {
        const int base = tok_base + 2 * tig - lo;
        const uint32_t cnt = static_cast<uint32_t>(ctx - lo);
        auto vis = [&](int d) { return static_cast<uint32_t>(base + d) < cnt; };
        keep_lo = (vis(0) ? 0x0000FFFFu : 0u) | (vis(1) ? 0xFFFF0000u : 0u);
        keep_hi = (vis(8) ? 0x0000FFFFu : 0u) | (vis(9) ? 0xFFFF0000u : 0u);
    }
    auto pv = [&](auto masked) {
        constexpr bool kMask = decltype(masked)::value;
        if constexpr (kFp8) {
            // e4m3 V straight from the raw tile.  The B operand pairs two
            // tokens of one dim; lane (g, tig) takes dims [g D/8, (g+1) D/8)
            // of V rows 2 tig, 2 tig + 1 (b0) and 2 tig + 8, 2 tig + 9 (b1), so
            // n-tile nt's column of this lane is dim g D/8 + nt.  O's n-tile nt
            // then holds dims 2 tig D/8 + nt and (2 tig + 1) D/8 + nt, which the
            // combine puts back in order.
            constexpr int W = D / 32;  // 32-bit words of a lane's slice of one row
            uint32_t r0[W], r1[W], r8[W], r9[W];
            const uint8_t* vb = vtile + g0 * (D / 8);
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
                if constexpr (kMask) {
                    b0a &= keep_lo;
                    b0b &= keep_lo;
                    b1a &= keep_hi;
                    b1b &= keep_hi;
                }
                mma_16816<true>(o[nt], pa, b0a, b1a);
                mma_16816<true>(o[nt + 1], pa, b0b, b1b);
            }
        } else {
            const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
            const int csel = lane >> 4;
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                const int chunk = 2 * j + csel;
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(v0, v1, v2, v3, vaddr + kv_off<D>(tok, chunk));
                if constexpr (kMask) {
                    v0 &= keep_lo;
                    v2 &= keep_lo;
                    v1 &= keep_hi;
                    v3 &= keep_hi;
                }
                mma_16816<kFp8>(o[2 * j], pa, v0, v1);
                mma_16816<kFp8>(o[2 * j + 1], pa, v2, v3);
            }
        }
    };
    // The skip pays on e4m3 tiles, where the ALU pipe sets the pace (the
    // conversions); bf16 tiles keep one masked loop (the second copy cost
    // the memory-bound bf16 kernel registers and time).
    if constexpr (kFp8) {
        if (edge)
            pv(std::true_type{});
        else
            pv(std::false_type{});
    } else {
        pv(std::true_type{});
    }
    (void)vaddr;
}

// kCluster: the chunks of one (sequence, KV head) form a thread-block cluster
// (grid x = cluster x = max_splits, so a chunk's cluster rank is blockIdx.x)
// and merge through distributed shared memory; otherwise through the
// workspace and a ticket.
template <int D, bool kFp8, bool kCluster, int kW>
__global__ void __launch_bounds__(kW * 32) decode_kernel(const DecodeArgs a,
                                                          const __grid_constant__ CUtensorMap kmap,
                                                          const __grid_constant__ CUtensorMap vmap) {
    using C = DecodeCfg<D, kFp8, kW>;
    constexpr int kThreads = kW * 32;
    constexpr int KSTEPS = D / 16;   // k-steps of Q.K^T
    constexpr int NTILES = D / 8;    // n-tiles of O
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bars[kW][C::kStages];
    __shared__ float s_m[kW][16];
    __shared__ float s_l[kW][16];
    __shared__ int s_flag;
    __shared__ __align__(8) uint64_t probe;  // test hook: a barrier nothing arrives on

    // Shared-memory set-up touches nothing the previous kernel writes: it
    // runs before the wait, while that kernel drains.
    if (threadIdx.x < kW * C::kStages) mbar_init(&bars[threadIdx.x / C::kStages][threadIdx.x % C::kStages], 1);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        s_flag = 0;
        if (a.inject_timeout) mbar_init(&probe, 1);
    }
    // With defer_wait the work overlaps the previous kernel and the
    // grid-dependency wait moves to the exit of CTA (0, 0, 0), which every
    // launch has: this grid then completes only after the previous one, so
    // kernels after this one see both, while every other CTA leaves as soon
    // as its work is done and frees its slot.  With early_kv the wait comes
    // after the lengths, the block ids and the first ring loads (the previous
    // kernel writes none of them) and before anything touches q, k_new, v_new
    // or an output; an exit before that point still waits.
    struct WaitAtExit {
        bool on;
        __device__ ~WaitAtExit() {
            if (on) pdl_wait();
        }
    };
    const bool early = a.early_kv != 0 && a.defer_wait == 0;
    WaitAtExit wait_at_exit{(a.defer_wait != 0 && is_first_cta()) || early};
    if (!a.defer_wait && !early) pdl_wait();
    // The next kernel may start once every CTA has triggered or exited, and
    // some CTA triggers only after its grid-dependency wait -- every CTA here,
    // the early-mode CTAs after their wait below (those without a chunk by
    // exiting; chunk 0 of each pair waits), CTA (0, 0, 0) of a deferred launch
    // by exiting after its wait at exit -- so the next kernel starts only once
    // this launch's predecessor has completed.
    if (!early && !(a.defer_wait != 0 && is_first_cta())) pdl_launch_dependents();
    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;

    // Without a window a chunk's blocks do not depend on the context length:
    // read this warp's block ids (below) while the length is still in
    // flight.  Entries past the sequence's end are read but unused.
    // Windowed cascade prefix pass: sequence seq reads the shared prefix of
    // its group (table row and length of the group; its own query position
    // is prefix + suffix_len - 1, so its window starts there).
    int row = seq;
    if (a.group_indptr) {
        int g_lo = 0, g_hi = a.num_groups - 1;
        while (g_lo < g_hi) {
            const int mid = (g_lo + g_hi + 1) >> 1;
            if (a.group_indptr[mid] <= seq)
                g_lo = mid;
            else
                g_hi = mid - 1;
        }
        row = g_lo;
    }
    const int32_t* bt = a.block_tables + static_cast<size_t>(row) * a.mbps;
    // Block ids of this warp's blocks: the k-th one in register k / 32 of
    // lane k % 32 (kIdRegs registers: up to 32 kIdRegs blocks per warp).
    int phys[C::kIdRegs];
#pragma unroll
    for (int r = 0; r < C::kIdRegs; ++r) phys[r] = 0;
    if (a.window <= 0) {
#pragma unroll
        for (int r = 0; r < C::kIdRegs; ++r) {
            const int lb = split * a.chunk_blocks + warp + (32 * r + lane) * kW;
            if ((32 * r + lane) * kW < a.chunk_blocks && lb < a.mbps) phys[r] = bt[lb];
        }
    }
    // A ring table of at most 32 entries holds every block a window can
    // touch: read all of it (lane k: entry k) while the length is in flight.
    const bool ring_lanes = a.ring > 0 && a.ring <= 32;
    int ring_id = 0;
    if (ring_lanes && lane < a.ring) ring_id = bt[lane];
    int ctx = a.context_lens[row];
    // the split plan (and the workspace) covers contexts up to max_ctx, which
    // the host checked against the table capacity
    bool clamped = false;
    if (ctx > a.max_ctx) {
        ctx = a.max_ctx;
        clamped = true;
    }
    // (errors are flagged after the grid-dependency wait: the error word is
    // written by earlier kernels too)
    auto flag_length = [&]() {
        if (clamped && threadIdx.x == 0 && split == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
    };
    if (!early) flag_length();
    int lo = (a.window > 0 && ctx > a.window) ? ctx - a.window : 0;
    if (a.group_indptr) {
        // the query at position ctx + suffix - 1 sees prefix keys t >= ctx + suffix - window
        lo = max(0, ctx + a.group_suffix_lens[seq] - a.window);
        if (lo >= ctx) ctx = 0;
    }
    if (ctx <= 0) {  // no visible key: o = 0, lse = -inf
        if (early) {
            pdl_wait();
            flag_length();
        }
        if (split == 0) {
            const size_t o0 = (static_cast<size_t>(seq) * a.hq + kvh * G) * D;
            for (int i = threadIdx.x; i < G * D; i += kThreads) {
                if (a.out_f32)
                    a.out_f32[o0 + i] = 0.f;
                else
                    static_cast<__nv_bfloat16*>(a.out)[o0 + i] = __float2bfloat16_rn(0.f);
            }
            if (a.lse_out && threadIdx.x < G)
                a.lse_out[static_cast<size_t>(seq) * a.hq + kvh * G + threadIdx.x] =
                    a.sinks ? a.sinks[kvh * G + threadIdx.x] : -INFINITY;
        }
        return;
    }
    const int first_blk = lo / kBlockSize;
    const int last_blk = (ctx - 1) / kBlockSize;
    const int nsplit = (last_blk - first_blk + a.chunk_blocks) / a.chunk_blocks;
    if (split >= nsplit) {
        // no chunk here.  In early mode the CTA leaves without waiting, so
        // its slot frees at once: chunk 0 of the same (sequence, KV head)
        // waits before it reads q or writes, so the grid still completes
        // after the previous kernel
        if (early) wait_at_exit.on = false;
        return;
    }
    const int b0 = first_blk + split * a.chunk_blocks;
    const int b1 = min(last_blk + 1, b0 + a.chunk_blocks);
    int my_n = (b1 - b0 > warp) ? (b1 - b0 - warp + kW - 1) / kW : 0;
    // a chunk longer than the warp's id registers hold (the host plans none):
    // flagged, and only the blocks whose ids it holds are read
    const bool too_long = my_n > 32 * C::kIdRegs;
    if (too_long) {
        if (!early && lane == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        my_n = 32 * C::kIdRegs;
    }

    fence_barrier_init();
    __syncthreads();

    // Physical block ids of this warp's blocks, checked: bit r of bad_ids
    // marks a bad id in register r (it reads block 0; the output is flagged).
    uint32_t bad_ids = 0;
#pragma unroll
    for (int r = 0; r < C::kIdRegs; ++r) {
        const int kb = 32 * r + lane;          // this lane's block in register r
        const int lb = b0 + warp + kb * kW;    // its logical block
        if (ring_lanes) {
            const int v = __shfl_sync(0xFFFFFFFFu, ring_id, kb < my_n ? lb % a.ring : 0);
            if (kb < my_n) phys[r] = v;
        }
        if (kb < my_n) {
            if (a.window > 0 && !ring_lanes) phys[r] = bt[a.ring > 0 ? lb % a.ring : lb];
            if (phys[r] < 0 || phys[r] >= a.num_blocks) {
                if (!early) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                phys[r] = 0;
                bad_ids |= 1u << r;
            }
        }
    }
    // the id of this warp's k-th block, read from its lane (every lane takes
    // part; k is the same in every lane, so all pick the same register)
    auto block_id = [&](int k) {
        int src = phys[0];
#pragma unroll
        for (int r = 1; r < C::kIdRegs; ++r)
            if ((k >> 5) == r) src = phys[r];
        return __shfl_sync(0xFFFFFFFFu, src, k & 31);
    };
    uint8_t* wbase = smem + warp * C::kWarpBytes;

    // Fused append: the warp that loads the sequence's last block writes the
    // new token into it first -- before its prologue when that block is one
    // of the first NSTAGE, else right after (the refill that loads it comes later).
    const int k_last = (last_blk - b0) / kW;
    const bool appender = a.k_new != nullptr && !clamped && split == nsplit - 1 &&
                          warp == (last_blk - b0) % kW && k_last < my_n;
    auto append = [&]() {
        const int pb = block_id(k_last);
        const bool bad = (__shfl_sync(0xFFFFFFFFu, bad_ids, k_last & 31) >> (k_last >> 5)) & 1u;
        if (!bad) append_new_token<D, kFp8>(a, seq, kvh, pb, ctx - 1, lane);
    };
    // Lane 0 issues the prologue; the shuffle reads lane k's id from lane 0's
    // point of view, so every lane takes part in it.
    auto load_stage = [&](int k) {
        const int pb = block_id(k);
        if (lane == 0 && k < my_n) {
            uint8_t* kdst = wbase + k * C::kStageBytes;
            uint8_t* vdst = kdst + C::kTileBytes;
            mbar_arrive_expect_tx(&bars[warp][k], C::kStageBytes);
            load_tile<kFp8>(kdst, &kmap, &bars[warp][k], kvh, pb);
            load_tile<kFp8>(vdst, &vmap, &bars[warp][k], kvh, pb);
        }
    };
    const bool append_first = appender && k_last < C::kStages;  // the new token's block is in the prologue
    if (!early) {
        if (append_first) append();
#pragma unroll
        for (int k = 0; k < C::kStages; ++k) load_stage(k);
    } else {
        // every stage but the one the new token goes into, then the wait
#pragma unroll
        for (int k = 0; k < C::kStages; ++k)
            if (!(append_first && k == k_last)) load_stage(k);
        pdl_wait();
        pdl_launch_dependents();
        flag_length();
        if (too_long && lane == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        if (__any_sync(0xFFFFFFFFu, bad_ids != 0)) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
        }
        if (append_first) {
            append();
            load_stage(k_last);
        }
    }
    if (appender && k_last >= C::kStages) append();

    // Q fragments (A operand, rows = heads of the group, zero-padded to 16).
    const int g0 = lane >> 2;
    const int tig = lane & 3;
    uint32_t qa[KSTEPS][4];
    load_q<D>(a, seq, kvh, (a.k_new != nullptr && a.cos_sin != nullptr && !clamped) ? ctx - 1 : -1, lane, qa);
    {
        if constexpr (kFp8) {
            // e4m3 pools: K fragments come straight from the raw tile, lane
            // (g, tig) reading its rows' bytes [tig D/4, (tig+1) D/4), so
            // k-step kk of that lane holds dims tig D/4 + 4 kk + {0,1} (k =
            // 2 tig, 2 tig + 1) and + {2,3} (k = 2 tig + 8, 2 tig + 9).  The
            // dot product is a sum over dims, so q takes the same order:
            // stage the rows in shared memory and read them back permuted.
            uint8_t* qs = wbase + C::kStages * C::kStageBytes;  // the f16 V buffer, free until the loop
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    const int row = g0 + ((part & 1) ? 8 : 0);
                    const int col = kk * 16 + 2 * tig + ((part & 2) ? 8 : 0);
                    *reinterpret_cast<uint32_t*>(qs + (row * D + col) * 2) = qa[kk][part];
                }
            __syncwarp();
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    const int row = g0 + ((part & 1) ? 8 : 0);
                    const int dim = tig * (D / 4) + 4 * kk + ((part & 2) ? 2 : 0);
                    const uint32_t v = *reinterpret_cast<const uint32_t*>(qs + (row * D + dim) * 2);
                    qa[kk][part] = pack2<true>(bf16_lo(v), bf16_hi(v));
                }
            __syncwarp();
        }
    }
    float scale_log2 = a.sm_scale * 1.4426950408889634f;
    if constexpr (kFp8) scale_log2 *= a.k_scale[kvh];

    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const bool hi_rows = G > 8;  // else each lane's second row (g0 + 8) is padding: its P stays 0
    float o[NTILES][4];
#pragma unroll
    for (int nt = 0; nt < NTILES; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;


    bool failed = false;
    const bool inject = a.inject_timeout != 0 && warp == 0 && is_first_cta();
    int k = 0;
    // the same loop for groups of more than 8 heads (rows 8-15 real) or not
    auto run_blocks = [&](auto hi) {
        for (; k < my_n; ++k) {
            const int st = k % C::kStages;
            const uint32_t ph = (k / C::kStages) & 1;
            const bool ready = __all_sync(
                0xFFFFFFFFu, (inject && k == 0) ? mbar_wait(&probe, 0, 1000ull * a.inject_limit_us)
                                                : mbar_wait(&bars[warp][st], ph));
            if (!ready) {
                failed = true;
                return;
            }
            const uint8_t* ktile = wbase + st * C::kStageBytes;
            attend_block<D, kFp8, decltype(hi)::value>(qa, o, m_run, l_run, ktile, ktile + C::kTileBytes,
                                                         lane, (b0 + warp + k * kW) * kBlockSize, lo, ctx,
                                                         scale_log2);
            __syncwarp();
            // refill this stage with the block NSTAGE ahead.  The stage was only
            // read, by this warp's loads, whose values the MMAs above consumed
            // before the __syncwarp: no proxy fence is needed before the copy
            // overwrites it (measured 2 % faster on the e4m3 decode without it)
            const int kn = k + C::kStages;
            const int pb = block_id(kn);
            if (lane == 0 && kn < my_n) {
                uint8_t* kdst = wbase + st * C::kStageBytes;
                uint8_t* vdst = kdst + C::kTileBytes;
                mbar_arrive_expect_tx(&bars[warp][st], C::kStageBytes);
                load_tile<kFp8>(kdst, &kmap, &bars[warp][st], kvh, pb);
                load_tile<kFp8>(vdst, &vmap, &bars[warp][st], kvh, pb);
            }
        }
    };
    if (hi_rows)
        run_blocks(std::true_type{});
    else
        run_blocks(std::false_type{});
    if (failed) {
        // drain the loads still in flight -- the stage that gave up and the
        // ones after it (bounded) -- so that no copy lands after exit, then report
        for (int kk = k; kk < min(my_n, k + C::kStages); ++kk)
            (void)mbar_wait(&bars[warp][kk % C::kStages], (kk / C::kStages) & 1);
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
    const size_t pair = static_cast<size_t>(seq) * a.hkv + kvh;
    // per row, once: the warps' weights 2^(m_w - M) / L (v_scale folded in)
    // replace s_m, and the row's lse goes to s_l[0]
    if (threadIdx.x < 16) {
        const int r = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kW; ++w) M = fmaxf(M, s_m[w][r]);
        float f[kW];
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            f[w] = s_m[w][r] == -INFINITY ? 0.f : fast_exp2(s_m[w][r] - M);
            L += f[w] * s_l[w][r];
        }
        // a failed chunk contributes nothing: weight 0, lse = -inf
        float inv = L > 0.f && !cta_failed ? (kFp8 ? a.v_scale[kvh] : 1.f) / L : 0.f;
        // a failed chunk's state is excluded from the merge by lse = -inf
        float lse = L > 0.f && !cta_failed ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
        if (a.sinks && nsplit == 1 && r < G) {
            // the sink joins the normaliser: lse' = ln(e^lse + e^s), o scaled by e^(lse - lse')
            const float sk = a.sinks[kvh * G + r];
            const float hi = fmaxf(lse, sk);
            const float lse2 = hi == -INFINITY ? -INFINITY : hi + __logf(__expf(lse - hi) + __expf(sk - hi));
            inv *= lse == -INFINITY ? 0.f : __expf(lse - lse2);
            lse = lse2;
        }
#pragma unroll
        for (int w = 0; w < kW; ++w) s_m[w][r] = f[w] * inv;
        s_l[0][r] = lse;
    }
    __syncthreads();
    {
        for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
            const int r = idx / D;
            const int d = idx % D;
            float ov = 0.f;
            if (!cta_failed) {
#pragma unroll
                for (int w = 0; w < kW; ++w) ov += s_m[w][r] * comb[(w * 16 + r) * C::kCombStride + d];
            }
            if (nsplit == 1) {
                const size_t oi = (static_cast<size_t>(seq) * a.hq + kvh * G + r) * D + d;
                if (a.out_f32)
                    a.out_f32[oi] = ov;
                else
                    static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(ov);
                if (a.lse_out && d == 0) a.lse_out[static_cast<size_t>(seq) * a.hq + kvh * G + r] = s_l[0][r];
            } else if (kCluster) {
                // this chunk's state stays in shared memory, in place of warp 0's rows
                comb[r * C::kCombStride + d] = ov;
            } else {
                const size_t prow = (pair * a.max_splits + split) * G + r;
                a.part_o[prow * D + d] = ov;
                if (d == 0) a.part_lse[prow] = s_l[0][r];
            }
        }
    }
    if (nsplit == 1) return;
    // the 2-warp variant runs one-chunk plans only; the merges below assume 4 warps
    if constexpr (kW < kWarps) return;

    if constexpr (kCluster) {
        // ---- cluster merge: chunk c of the pair holds o_c (rows of warp 0's
        // slice of comb) and lse_c (s_l[0]) in its shared memory
        cluster_sync();
        float* wts = comb + 16 * C::kCombStride;  // warp 1's slice, free now: [chunk][16]
        float* rowM = wts + kMaxClusterSplits * 16;
        float* rowW = rowM + 16;
        if (threadIdx.x < 16) {
            const int r = threadIdx.x;
            float l[kMaxClusterSplits];
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxClusterSplits; ++c) {
                l[c] = c < nsplit ? ld_cluster_f32(cluster_map(smem_u32(&s_l[0][r]), c)) : -INFINITY;
                M = fmaxf(M, l[c]);
            }
            float W = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxClusterSplits; ++c) {
                const float wv = l[c] == -INFINITY ? 0.f : __expf(l[c] - M);
                wts[c * 16 + r] = wv;
                W += wv;
            }
            if (a.sinks && r < G && M != -INFINITY) W += __expf(a.sinks[kvh * G + r] - M);
            rowM[r] = M;
            rowW[r] = W;
        }
        __syncthreads();
        // this chunk merges its share of the G x D output, in float4 slots
        constexpr int kSlotsPerRow = D / 4;
        const int total = G * kSlotsPerRow;
        const int s_lo = split * total / nsplit;
        const int s_hi = (split + 1) * total / nsplit;
        for (int slot = s_lo + threadIdx.x; slot < s_hi; slot += kThreads) {
            const int r = slot / kSlotsPerRow;
            const int c4 = slot % kSlotsPerRow;
            const uint32_t local = smem_u32(comb + r * C::kCombStride + c4 * 4);
            float4 v[kMaxClusterSplits];
#pragma unroll
            for (int c = 0; c < kMaxClusterSplits; ++c)
                if (c < nsplit) v[c] = ld_cluster_f32x4(cluster_map(local, c));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kMaxClusterSplits; ++c) {
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
            const size_t oi = (static_cast<size_t>(seq) * a.hq + kvh * G + r) * D + c4 * 4;
            if (a.out_f32) {
                *reinterpret_cast<float4*>(a.out_f32 + oi) =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            } else {
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) =
                    make_uint2(pack2<false>(acc.x * inv, acc.y * inv), pack2<false>(acc.z * inv, acc.w * inv));
            }
            if (a.lse_out && c4 == 0)
                a.lse_out[static_cast<size_t>(seq) * a.hq + kvh * G + r] =
                    W > 0.f ? rowM[r] + __logf(W) : -INFINITY;
        }
        cluster_sync();  // no chunk exits while a peer may still read its shared memory
        return;
    }

    // ---- ticket: the last chunk of this (sequence, KV head) merges
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_flag = static_cast<int>(atomicAdd(&a.counters[pair], 1u));
    __syncthreads();
    if (s_flag != nsplit - 1) return;
    __threadfence();
    // weights per (split, row) in shared memory: wts[split][16], then M, W per row
    float* wts = reinterpret_cast<float*>(smem);
    float* rowM = wts + a.max_splits * 16;
    float* rowW = rowM + 16;
    {
        const int r = threadIdx.x >> 3;  // 16 rows x 8 threads
        const int sub = threadIdx.x & 7;
        float M = -INFINITY;
        if (r < G)
            for (int i = sub; i < nsplit; i += 8)
                M = fmaxf(M, __ldcg(a.part_lse + (pair * a.max_splits + i) * G + r));
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
        float W = 0.f;
        if (r < G)
            for (int i = sub; i < nsplit; i += 8) {
                const float l = __ldcg(a.part_lse + (pair * a.max_splits + i) * G + r);
                const float wv = l == -INFINITY ? 0.f : __expf(l - M);
                wts[i * 16 + r] = wv;
                W += wv;
            }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) W += __shfl_xor_sync(0xFFFFFFFFu, W, off);
        if (sub == 0) {
            // a sink joins the normaliser (M is finite: every split has keys)
            if (a.sinks && r < G) W += __expf(a.sinks[kvh * G + r] - M);
            rowM[r] = M;
            rowW[r] = W;
        }
    }
    __syncthreads();
    // Each thread owns float4 slots (row, 4 columns); the loads of all splits
    // are independent, four in flight per slot, so the merge costs a few L2
    // round trips rather than one per split.
    constexpr int kSlotsPerRow = D / 4;
    const float4* po = reinterpret_cast<const float4*>(a.part_o);
    for (int slot = threadIdx.x; slot < G * kSlotsPerRow; slot += kThreads) {
        const int r = slot / kSlotsPerRow;
        const int c4 = slot % kSlotsPerRow;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int i = 0;
        for (; i + 4 <= nsplit; i += 4) {
            float4 v[4];
            float w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                w[u] = wts[(i + u) * 16 + r];
                v[u] = __ldcg(po + ((pair * a.max_splits + i + u) * G + r) * kSlotsPerRow + c4);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (w[u] != 0.f) {
                    acc.x += w[u] * v[u].x;
                    acc.y += w[u] * v[u].y;
                    acc.z += w[u] * v[u].z;
                    acc.w += w[u] * v[u].w;
                }
            }
        }
        for (; i < nsplit; ++i) {
            const float w = wts[i * 16 + r];
            const float4 v = __ldcg(po + ((pair * a.max_splits + i) * G + r) * kSlotsPerRow + c4);
            if (w != 0.f) {
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
        }
        const float W = rowW[r];
        const float inv = W > 0.f ? 1.f / W : 0.f;
        const size_t oi = (static_cast<size_t>(seq) * a.hq + kvh * G + r) * D + c4 * 4;
        if (a.out_f32) {
            *reinterpret_cast<float4*>(a.out_f32 + oi) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) =
                make_uint2(pack2<false>(acc.x * inv, acc.y * inv), pack2<false>(acc.z * inv, acc.w * inv));
        }
        if (a.lse_out && c4 == 0)
            a.lse_out[static_cast<size_t>(seq) * a.hq + kvh * G + r] =
                W > 0.f ? rowM[r] + __logf(W) : -INFINITY;
    }
    if (threadIdx.x == 0) a.counters[pair] = 0u;
}

template <int D, bool kFp8, bool kCluster, int kW>
cudaError_t launch_decode_v(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
    using C = DecodeCfg<D, kFp8, kW>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert((kMaxClusterSplits + 2) * 16 <= 16 * C::kCombStride, "cluster merge scratch");
    auto kern = decode_kernel<D, kFp8, kCluster, kW>;
    // The shared-memory opt-in is a per-device function attribute: set it on
    // the first launch on each device (never inside a stream capture).
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid(a.max_splits, a.hkv, a.num_seqs);
    return launch_pdl_cluster(kern, grid, dim3(kW * 32), C::kSmemBytes, stream,
                              kCluster ? static_cast<unsigned>(a.max_splits) : 1u, a, kmap, vmap);
}

template <int D, bool kFp8>
cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
    // A windowed plan of one chunk per sequence has a few blocks per CTA:
    // 2-warp CTAs, more of them resident, keep such a layer to one wave.
    // (Each lane of a 2-warp CTA holds one block id of its warp: at most 32
    // blocks per warp.)
    if (a.window > 0 && a.max_splits == 1 && a.chunk_blocks <= 2 * 32)
        return launch_decode_v<D, kFp8, false, 2>(a, kmap, vmap, stream);
    if (a.max_splits >= 2 && a.max_splits <= kMaxClusterSplits)
        return launch_decode_v<D, kFp8, true, kWarps>(a, kmap, vmap, stream);
    return launch_decode_v<D, kFp8, false, kWarps>(a, kmap, vmap, stream);
}

}  // namespace

bool decode_uses_tickets(int splits) { return splits > kMaxClusterSplits; }

int decode_smem_bytes(int d, int fp8) {
    if (d == 64) return fp8 ? DecodeCfg<64, true>::kSmemBytes : DecodeCfg<64, false>::kSmemBytes;
    return fp8 ? DecodeCfg<128, true>::kSmemBytes : DecodeCfg<128, false>::kSmemBytes;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream) {
    if (a.d == 64) {
        return a.fp8 ? launch_decode_t<64, true>(a, kmap, vmap, stream)
                     : launch_decode_t<64, false>(a, kmap, vmap, stream);
    }
    return a.fp8 ? launch_decode_t<128, true>(a, kmap, vmap, stream)
                 : launch_decode_t<128, false>(a, kmap, vmap, stream);
}

}  // namespace pkv
