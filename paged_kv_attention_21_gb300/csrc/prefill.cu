// prefill.cu -- ragged, causal, chunked-prefill attention over cached prefixes.
//
// What it computes (infer-lab, "Technique" table: chunked prefill slices a
// long prompt; llm-infer, "What It Does": ragged batched prefill; the
// online-softmax tiling of FlashAttention-2, llm-infer "References"):
// sequence s has q_len new query tokens whose K/V are already in the paged
// cache after a cached prefix; query i sits at position
// p_i = kv_len - q_len + i and attends keys t <= p_i (and t > p_i - W with a
// window), read block by block through the block table.
//
// Work decomposition.  One CTA owns (sequence, KV head, query tile).  A query
// tile packs QT consecutive tokens x the G heads of one KV group into 64
// rows (row r -> token r / G, head r % G), so one read of a K/V tile serves
// every query head that shares it.  A producer warp streams K/V tiles of 64
// keys (4 blocks) through a 3-stage TMA ring (full/empty mbarriers); four
// consumer warps each own 16 rows and run
//     S[16 x 64] = Q . K^T  -> causal/window mask -> online softmax
//     O[16 x D] += P . V
// on mma.sync m16n8k16 bf16 with fp32 accumulation.  KV tiles wholly
// visible to a warp skip the mask; tiles past the causal diagonal of the
// whole CTA are never loaded.
//
// Roofline: tensor pipe -- 4*D*G flops per (query token, key) pair against
// K/V bytes that stay in L2 across the query tiles of a sequence.
#include "common.cuh"
#include "internal.h"

namespace pkv {

namespace {

constexpr int kConsumers = 4;
constexpr int kPThreads = (kConsumers + 1) * 32;
constexpr int kRows = kConsumers * 16;
constexpr int kKvTile = 64;                       // keys per stage
constexpr int kBlocksPerTile = kKvTile / kBlockSize;

template <int D>
struct PrefillCfg {
    static constexpr int kStages = 3;
    static constexpr int kBlockTileBytes = kBlockSize * D * 2;        // one block, one head, bf16
    static constexpr int kHalfBytes = kBlockTileBytes * kBlocksPerTile;  // K (or V) of a stage
    static constexpr int kStageBytes = 2 * kHalfBytes;
    static constexpr int kBoxes = D / 64;
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
};

template <int D>
__global__ void __launch_bounds__(kPThreads) prefill_kernel(const PrefillArgs a,
                                                            const __grid_constant__ CUtensorMap kmap,
                                                            const __grid_constant__ CUtensorMap vmap) {
    using C = PrefillCfg<D>;
    constexpr int KSTEPS = D / 16;
    constexpr int NTILES = D / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full[C::kStages];
    __shared__ __align__(8) uint64_t empty[C::kStages];
    __shared__ int s_fail;

    pdl_wait();
    pdl_launch_dependents();
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int G = a.group;
    const int QT = a.q_tile;
    const int q0 = a.qo_indptr[seq];
    const int q_len = a.qo_indptr[seq + 1] - q0;
    if (q0 < 0 || q_len < 0 || q0 + q_len > a.total_q) {  // rows outside q / out
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_POSITION);
        return;
    }
    int kv_len = a.kv_lens[seq];
    const int cap = a.mbps * kBlockSize;
    if (kv_len > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        kv_len = cap;
    }
    const int ntiles = (q_len + QT - 1) / QT;
    if (static_cast<int>(blockIdx.x) >= ntiles) return;
    const int qt = ntiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
    const int tok0 = qt * QT;                                   // first token of the tile
    const int ntok = min(QT, q_len - tok0);
    const int off = kv_len - q_len;                             // position of token 0
    const int pos_min = off + tok0;
    const int pos_max = off + tok0 + ntok - 1;
    // key range this CTA may need
    int key_hi = a.causal ? min(pos_max, kv_len - 1) : kv_len - 1;
    int key_lo = 0;
    if (a.window > 0) key_lo = max(0, pos_min - a.window + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumers);
        }
        s_fail = 0;
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    fence_barrier_init();
    __syncthreads();

    const int t_begin = key_lo / kKvTile;
    const int t_end = key_hi >= key_lo ? key_hi / kKvTile + 1 : t_begin;
    const int n_tiles = t_end - t_begin;
    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.mbps;
    const int nblk_seq = (kv_len + kBlockSize - 1) / kBlockSize;

    if (warp == kConsumers) {
        // ------------------------------------------------------ producer
        int ids = 0;  // lane l holds block id (round base + l)
        int base = -1;
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i % C::kStages;
            const uint32_t ph = ((i / C::kStages) & 1) ^ 1;
            const int blk0 = (t_begin + i) * kBlocksPerTile;
            if (base < 0 || blk0 + kBlocksPerTile > base + 32) {
                base = blk0;
                ids = 0;
                if (base + lane < nblk_seq) {
                    ids = bt[base + lane];
                    if (ids < 0 || ids >= a.num_blocks) {
                        flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                        ids = 0;
                    }
                }
            }
            int pb[kBlocksPerTile];
#pragma unroll
            for (int b = 0; b < kBlocksPerTile; ++b) pb[b] = __shfl_sync(0xFFFFFFFFu, ids, blk0 - base + b);
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&empty[st], ph);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) {
                    flag_error(a.err, PKV_DEVERR_TIMEOUT);
                    atomicOr(&s_fail, 1);
                    // never leave the consumers waiting on a stage with no load
                    for (int j = i; j < min(n_tiles, i + C::kStages); ++j) mbar_arrive(&full[j % C::kStages]);
                }
                break;
            }
            if (lane == 0) {
                int nvalid = 0;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) nvalid += (blk0 + b < nblk_seq) ? 1 : 0;
                uint8_t* kdst = smem + st * C::kStageBytes;
                uint8_t* vdst = kdst + C::kHalfBytes;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&full[st], nvalid * 2 * C::kBlockTileBytes);
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    if (blk0 + b >= nblk_seq) break;
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx) {
                        tma_load_4d(kdst + b * C::kBlockTileBytes + bx * 2048, &kmap, &full[st], bx * 64, 0,
                                    kvh, pb[b]);
                        tma_load_4d(vdst + b * C::kBlockTileBytes + bx * 2048, &vmap, &full[st], bx * 64, 0,
                                    kvh, pb[b]);
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int g0 = lane >> 2;
    const int tig = lane & 3;
    const int r0 = warp * 16 + g0;
    const int r1 = r0 + 8;
    const int t0 = r0 / G, t1 = r1 / G;
    const bool row0_ok = t0 < ntok && r0 < QT * G;
    const bool row1_ok = t1 < ntok && r1 < QT * G;
    const int pos0 = off + tok0 + t0;
    const int pos1 = off + tok0 + t1;
    // warp-wide bounds for the fully-visible test
    int wpos_min = 0x7FFFFFFF, wpos_max = -1;
    {
        const int lo_row = warp * 16, hi_row = min(warp * 16 + 15, QT * G - 1);
        for (int r = lo_row; r <= hi_row; ++r) {
            const int t = r / G;
            if (t < ntok) {
                wpos_min = min(wpos_min, off + tok0 + t);
                wpos_max = max(wpos_max, off + tok0 + t);
            }
        }
    }
    const bool warp_active = wpos_max >= 0;

    uint32_t qa[KSTEPS][4];
    {
        const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const int row = (part & 1) ? r1 : r0;
            const bool ok = (part & 1) ? row1_ok : row0_ok;
            const __nv_bfloat16* qrow =
                qb + (static_cast<size_t>(q0 + tok0 + row / G) * a.hq + kvh * G + row % G) * D;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int col = kk * 16 + 2 * tig + ((part & 2) ? 8 : 0);
                qa[kk][part] = ok ? *reinterpret_cast<const uint32_t*>(qrow + col) : 0u;
            }
        }
    }
    const float scale_log2 = a.sm_scale * 1.4426950408889634f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[NTILES][4];
#pragma unroll
    for (int nt = 0; nt < NTILES; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    bool failed = false;
    for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait(&full[st], ph));
        if (!ready || s_fail) {
            failed = true;
            break;
        }
        const int k0 = (t_begin + i) * kKvTile;
        // tiles this warp cannot see at all are skipped (still released)
        bool skip = !warp_active;
        if (a.causal && k0 > wpos_max) skip = true;
        if (a.window > 0 && k0 + kKvTile - 1 <= wpos_min - a.window) skip = true;
        if (!skip) {
            const bool full_vis = (!a.causal || k0 + kKvTile - 1 <= wpos_min) &&
                                  (k0 + kKvTile <= kv_len) &&
                                  (a.window <= 0 || k0 > wpos_max - a.window);
            const uint32_t kaddr = smem_u32(smem + st * C::kStageBytes);
            const uint32_t vaddr = kaddr + C::kHalfBytes;
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
            {
                const int tok = (lane & 7) + ((lane >> 4) << 3);
                const int csel = (lane >> 3) & 1;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        const int chunk = 2 * kk + csel;
                        uint32_t b00, b01, b10, b11;
                        ldmatrix_x4(b00, b01, b10, b11,
                                    kaddr + b * C::kBlockTileBytes + (chunk >> 3) * 2048 +
                                        sw128(tok, chunk & 7));
                        mma_16816<false>(s[2 * b], qa[kk], b00, b01);
                        mma_16816<false>(s[2 * b + 1], qa[kk], b10, b11);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = s[n][e] * scale_log2;
                    if (!full_vis) {
                        const int t = k0 + n * 8 + 2 * tig + (e & 1);
                        const int pos = (e < 2) ? pos0 : pos1;
                        const bool vis = t < kv_len && (!a.causal || t <= pos) &&
                                         (a.window <= 0 || t > pos - a.window);
                        if (!vis) x = -INFINITY;
                    }
                    s[n][e] = x;
                }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
                mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
            }
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
            float ls0 = 0.f, ls1 = 0.f;
            uint32_t pa[4][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const float p0 = fast_exp2(s[n][0] - mu0);
                const float p1 = fast_exp2(s[n][1] - mu0);
                const float p2 = fast_exp2(s[n][2] - mu1);
                const float p3 = fast_exp2(s[n][3] - mu1);
                ls0 += p0 + p1;
                ls1 += p2 + p3;
                // n-tile n covers keys 8n..8n+7: k-step n/2, low or high half
                pa[n >> 1][(n & 1) ? 2 : 0] = pack2<false>(p0, p1);
                pa[n >> 1][(n & 1) ? 3 : 1] = pack2<false>(p2, p3);
            }
            l_run[0] = l_run[0] * al0 + ls0;
            l_run[1] = l_run[1] * al1 + ls1;
            if (__any_sync(0xFFFFFFFFu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int nt = 0; nt < NTILES; ++nt) {
                    o[nt][0] *= al0;
                    o[nt][1] *= al0;
                    o[nt][2] *= al1;
                    o[nt][3] *= al1;
                }
            }
            {
                const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
                const int csel = lane >> 4;
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b) {
                    uint32_t keep_lo = 0xFFFFFFFFu, keep_hi = 0xFFFFFFFFu;
                    const int tb = k0 + b * kBlockSize + 2 * tig;
                    if (k0 + kKvTile > kv_len) {  // keys past kv_len: zero V
                        keep_lo = (tb < kv_len ? 0x0000FFFFu : 0u) | (tb + 1 < kv_len ? 0xFFFF0000u : 0u);
                        keep_hi = (tb + 8 < kv_len ? 0x0000FFFFu : 0u) | (tb + 9 < kv_len ? 0xFFFF0000u : 0u);
                    }
#pragma unroll
                    for (int j = 0; j < D / 16; ++j) {
                        const int chunk = 2 * j + csel;
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(v0, v1, v2, v3,
                                          vaddr + b * C::kBlockTileBytes + (chunk >> 3) * 2048 +
                                              sw128(tok, chunk & 7));
                        v0 &= keep_lo;
                        v2 &= keep_lo;
                        v1 &= keep_hi;
                        v3 &= keep_hi;
                        mma_16816<false>(o[2 * j], pa[b], v0, v1);
                        mma_16816<false>(o[2 * j + 1], pa[b], v2, v3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (failed) {
        if (lane == 0) flag_error(a.err, PKV_DEVERR_TIMEOUT);
        return;
    }

    l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], 1);
    l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], 2);
    l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], 1);
    l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], 2);
    const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
    const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out);
    const size_t orow0 = (static_cast<size_t>(q0 + tok0 + t0) * a.hq + kvh * G + r0 % G) * D;
    const size_t orow1 = (static_cast<size_t>(q0 + tok0 + t1) * a.hq + kvh * G + r1 % G) * D;
#pragma unroll
    for (int nt = 0; nt < NTILES; ++nt) {
        const int col = nt * 8 + 2 * tig;
        if (row0_ok)
            *reinterpret_cast<uint32_t*>(ob + orow0 + col) = pack2<false>(o[nt][0] * inv0, o[nt][1] * inv0);
        if (row1_ok)
            *reinterpret_cast<uint32_t*>(ob + orow1 + col) = pack2<false>(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (a.lse_out && tig == 0) {
        const float ln2 = 0.6931471805599453f;
        if (row0_ok)
            a.lse_out[static_cast<size_t>(q0 + tok0 + t0) * a.hq + kvh * G + r0 % G] =
                l_run[0] > 0.f ? (m_run[0] + __log2f(l_run[0])) * ln2 : -INFINITY;
        if (row1_ok)
            a.lse_out[static_cast<size_t>(q0 + tok0 + t1) * a.hq + kvh * G + r1 % G] =
                l_run[1] > 0.f ? (m_run[1] + __log2f(l_run[1])) * ln2 : -INFINITY;
    }
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
    using C = PrefillCfg<D>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    auto kern = prefill_kernel<D>;
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
    dim3 grid(a.max_qtiles, a.hkv, a.num_seqs);
    return launch_pdl(kern, grid, dim3(kPThreads), C::kSmemBytes, stream, a, kmap, vmap);
}

}  // namespace

int prefill_q_tile(int group) { return group >= 1 && group <= kRows ? kRows / group : 0; }

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
    return a.d == 64 ? launch_prefill_t<64>(a, kmap, vmap, stream)
                     : launch_prefill_t<128>(a, kmap, vmap, stream);
}

}  // namespace pkv
