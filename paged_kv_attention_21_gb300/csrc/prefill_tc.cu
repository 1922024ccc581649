// prefill_tc.cu -- ragged, causal, chunked-prefill attention over cached
// prefixes on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes (infer-lab, "Technique" table: chunked prefill; llm-infer,
// "What It Does": ragged batched prefill; FlashAttention-2's online softmax,
// llm-infer "References"): sequence s has q_len new query tokens, already
// appended to the paged cache behind a cached prefix; query i sits at
// position p_i = kv_len - q_len + i and attends keys t <= p_i (and
// t > p_i - W with a window), gathered block by block through the block table.
//
// One CTA owns (sequence, KV head, query tile).  The tile packs QT = 128 / G
// consecutive query tokens x the G heads of one KV group into M = 128 rows
// (row r -> token r / G, head r % G), so each K/V tile read serves the whole
// group.  Warp roles:
//   warp 0      TMA producer: the Q tile once (3-D tensor map over q), then
//               K and V tiles of 128 keys (8 blocks) into separate rings
//               (2 stages each; K frees at S completion, V at PV completion);
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               S buffers, then O += P_{j-1} V_{j-1} into the TMEM O
//               accumulator -- so S_{j+1} runs on the tensor pipe while the
//               softmax warps work on S_j;
//   warps 2..9  softmax, two threads per row (its TMEM lane; 64 key columns
//               each, row maxima exchanged in shared memory): masked row max,
//               lazy rescale of O only when the max grows by more than 2^8,
//               P = 2^(x - m) (fp32 exp2, packed to bf16) written to shared
//               memory in the 128-byte-swizzled K-major layout the MMA reads,
//               and the final 1/l normalisation and bf16 store.
// Operands: Q, K (K-major, SW128) and P (K-major, SW128) via shared-memory
// descriptors; V is read MN-major (head_dim contiguous), as stored.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTcM = 128;                         // query rows per tile
constexpr int kTcN = 128;                         // keys per KV tile
constexpr int kTcBlocks = kTcN / kBlockSize;      // 8 blocks per KV tile
constexpr int kTcWarps = 10;  // producer, MMA issuer, 8 softmax warps (2 per row quadrant)
constexpr int kTcThreads = kTcWarps * 32;
constexpr float kRescaleThreshold = 8.0f;         // log2 of the largest stale-max factor

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;             // 64-column (128-byte) halves of a row
    static constexpr int kHalfBytes = 128 * 128;       // 128 rows x 128 bytes
    static constexpr int kQBytes = kHalves * kHalfBytes;
    static constexpr int kKBytes = kHalves * kHalfBytes;  // 128 keys x D (K or V tile)
    static constexpr int kPBytes = 2 * kHalfBytes;        // 128 rows x 128 keys
    // K and V live in separate rings: a K stage frees as soon as its S = Q K^T
    // is done, so K runs a full tile further ahead of the MMA than V.
    static constexpr int kKStages = 2;
    static constexpr int kVStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffK = kOffP + kPBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    static constexpr int kBodyBytes = kOffV + kVStages * kKBytes;
    // at least 120 KB so that one CTA owns an SM (and all 512 TMEM columns)
    static constexpr int kSmemBytes = (kBodyBytes + 1024 > 120 * 1024) ? kBodyBytes + 1024 : 120 * 1024;
    static constexpr uint32_t kTmemCols = 512;            // S0 | S1 | O
    static constexpr uint32_t kColO = 256;
};

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
    using C = TcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t bar_q;
    __shared__ __align__(8) uint64_t bar_k[3];
    __shared__ __align__(8) uint64_t bar_k_empty[3];
    __shared__ __align__(8) uint64_t bar_v[2];
    __shared__ __align__(8) uint64_t bar_v_empty[2];
    __shared__ __align__(8) uint64_t bar_s_full[2];
    __shared__ __align__(8) uint64_t bar_s_free[2];
    __shared__ __align__(8) uint64_t bar_p_full;
    __shared__ __align__(8) uint64_t bar_o_done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ float s_red_max[2][2][kTcM];  // [tile parity][column half][row]
    __shared__ float s_red_sum[2][kTcM];     // [column half][row]
    __shared__ __align__(8) uint64_t bar_pair[4][3];  // per quadrant: tile parity 0/1, final

    pdl_wait();
    pdl_launch_dependents();
    const int kvh = blockIdx.y;
    const int seq = blockIdx.z;
    const int G = a.group;
    const int QT = a.q_tile;
    const int q0 = a.qo_indptr[seq];
    const int q_len = a.qo_indptr[seq + 1] - q0;
    if (q0 < 0 || q_len < 0 || q0 + q_len > a.total_q) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_POSITION);
        return;
    }
    int kv_len = a.kv_lens[seq];
    const int cap = a.mbps * kBlockSize;
    if (kv_len > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
        kv_len = cap;
    }
    const int ntiles_q = (q_len + QT - 1) / QT;
    if (static_cast<int>(blockIdx.x) >= ntiles_q) return;
    const int qt = ntiles_q - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
    const int tok0 = qt * QT;
    const int ntok = min(QT, q_len - tok0);
    const int off = kv_len - q_len;
    const int pos_min = off + tok0;
    const int pos_max = off + tok0 + ntok - 1;
    const int key_hi = a.causal ? min(pos_max, kv_len - 1) : kv_len - 1;
    const int key_lo = a.window > 0 ? max(0, pos_min - a.window + 1) : 0;
    const int t_begin = key_lo / kTcN;
    const int n_tiles = key_hi >= key_lo ? key_hi / kTcN + 1 - t_begin : 0;
    const int nblk_seq = (kv_len + kBlockSize - 1) / kBlockSize;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 1);
        for (int i = 0; i < C::kKStages; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_k_empty[i], 1);
        }
        for (int i = 0; i < C::kVStages; ++i) {
            mbar_init(&bar_v[i], 1);
            mbar_init(&bar_v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_s_full[i], 1);
            mbar_init(&bar_s_free[i], 8);
        }
        mbar_init(&bar_p_full, 8);
        for (int qd = 0; qd < 4; ++qd)
            for (int i = 0; i < 3; ++i) mbar_init(&bar_pair[qd][i], 64);
        mbar_init(&bar_o_done, 1);
        s_fail = 0;
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    if (warp == 1) {
        tc::tmem_alloc(&s_tmem, C::kTmemCols);
        tc::tmem_relinquish();
    }
    fence_barrier_init();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sP = smem + C::kOffP;
    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.mbps;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (n_tiles > 0) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_q, C::kHalves * 64 * 2 * G * QT);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d(sQ + h * C::kHalfBytes, &qmap, &bar_q, h * 64, kvh * G, q0 + tok0);
            }
            // order of loads: K_0, K_1, V_0, K_2, V_1, ... -- K one tile ahead of V
            int ids_prev = 0;
            for (int j = 0; j <= n_tiles; ++j) {
                int ids_cur = 0;
                if (j < n_tiles) {
                    const int blk0 = (t_begin + j) * kTcBlocks;
                    if (lane < kTcBlocks && blk0 + lane < nblk_seq) {
                        ids_cur = bt[blk0 + lane];
                        if (ids_cur < 0 || ids_cur >= a.num_blocks) {
                            flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                            ids_cur = 0;
                        }
                    }
                    const int st = j % C::kKStages;
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(&bar_k_empty[st], ((j / C::kKStages) & 1) ^ 1) ? 1 : 0;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    const int nvalid = min(kTcBlocks, nblk_seq - blk0);
                    uint8_t* sK = smem + C::kOffK + st * C::kKBytes;
                    int ids[kTcBlocks];
#pragma unroll
                    for (int b = 0; b < kTcBlocks; ++b) ids[b] = __shfl_sync(0xFFFFFFFFu, ids_cur, b);
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&bar_k[st], nvalid * kBlockSize * D * 2);
#pragma unroll
                        for (int b = 0; b < kTcBlocks; ++b) {
                            if (b >= nvalid) break;
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_load_4d(sK + h * C::kHalfBytes + b * 2048, &kmap, &bar_k[st], h * 64, 0,
                                            kvh, ids[b]);
                        }
                    }
                }
                if (j >= 1) {
                    const int i = j - 1;
                    const int st = i % C::kVStages;
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(&bar_v_empty[st], ((i / C::kVStages) & 1) ^ 1) ? 1 : 0;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    const int blk0 = (t_begin + i) * kTcBlocks;
                    const int nvalid = min(kTcBlocks, nblk_seq - blk0);
                    uint8_t* sV = smem + C::kOffV + st * C::kKBytes;
                    int ids[kTcBlocks];
#pragma unroll
                    for (int b = 0; b < kTcBlocks; ++b) ids[b] = __shfl_sync(0xFFFFFFFFu, ids_prev, b);
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(&bar_v[st], nvalid * kBlockSize * D * 2);
#pragma unroll
                        for (int b = 0; b < kTcBlocks; ++b) {
                            if (b >= nvalid) break;
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_load_4d(sV + h * C::kHalfBytes + b * 2048, &vmap, &bar_v[st], h * 64, 0,
                                            kvh, ids[b]);
                        }
                    }
                }
                ids_prev = ids_cur;
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTcM, kTcN, false, false);
        constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTcM, D, false, true);
        bool ok = n_tiles > 0 ? mbar_wait(&bar_q, 0) : true;
        ok = __all_sync(0xFFFFFFFFu, ok);
        for (int j = 0; ok && j <= n_tiles; ++j) {
            if (j < n_tiles) {
                const int st = j & 1;
                const int ks = j % C::kKStages;
                bool r1 = mbar_wait(&bar_k[ks], (j / C::kKStages) & 1);
                bool r2 = mbar_wait(&bar_s_free[st], ((j >> 1) & 1) ^ 1);
                if (!__all_sync(0xFFFFFFFFu, r1 && r2) || *reinterpret_cast<volatile int*>(&s_fail)) { ok = false; break; }
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint8_t* sK = smem + C::kOffK + ks * C::kKBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int h = kk >> 2;
                        const uint32_t ko = (kk & 3) * 32;
                        const uint64_t ad = tc::smem_desc(smem_u32(sQ + h * C::kHalfBytes) + ko, 16, 1024);
                        const uint64_t bd = tc::smem_desc(smem_u32(sK + h * C::kHalfBytes) + ko, 16, 1024);
                        tc::mma_bf16(tmem + st * kTcN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&bar_s_full[st]);
                    tc::commit(&bar_k_empty[ks]);  // this K tile is no longer needed
                }
                __syncwarp();
            }
            if (j >= 1) {
                const int i = j - 1;
                const int st = i % C::kVStages;
                bool r1 = mbar_wait(&bar_p_full, i & 1);
                bool r2 = mbar_wait(&bar_v[st], (i / C::kVStages) & 1);
                if (!__all_sync(0xFFFFFFFFu, r1 && r2) || *reinterpret_cast<volatile int*>(&s_fail)) { ok = false; break; }
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint8_t* sV = smem + C::kOffV + st * C::kKBytes;
#pragma unroll
                    for (int kk = 0; kk < kTcN / 16; ++kk) {
                        const int h = kk >> 2;
                        const uint32_t ko = (kk & 3) * 32;
                        const uint64_t ad = tc::smem_desc(smem_u32(sP + h * C::kHalfBytes) + ko, 16, 1024);
                        // V, MN-major: 16 keys per k-step = 2 groups of 8 rows (SBO 1024);
                        // the two 64-column halves of head_dim are C::kHalfBytes apart (LBO)
                        const uint64_t bd = tc::smem_desc(smem_u32(sV) + kk * 2048, C::kHalfBytes, 1024);
                        tc::mma_bf16(tmem + C::kColO, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(&bar_o_done);
                    tc::commit(&bar_v_empty[st]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            atomicOr(&s_fail, 1);
        }
    } else {
        // -------------------------------------------------------------- softmax
        // Two warps share each row quadrant: warp w (2..9) reads TMEM lanes of
        // quadrant w % 4 and owns key columns [64h, 64h + 64) and O columns
        // [h D/2, (h+1) D/2) with h = (w - 2) / 4.  The pair exchanges row maxima
        // through shared memory on a named barrier; row sums stay per half.
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;          // key / O column half
        const int r = quad * 32 + lane;            // the row this thread owns
        const int t = r / G;
        const bool row_ok = r < QT * G && t < ntok;
        const int pos = off + tok0 + t;
        const float scale_log2 = a.sm_scale * 1.4426950408889634f;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const int sm_tid = (warp - 2) * 32 + lane;  // 0..255
        // the two warps of this quadrant meet on an mbarrier (bounded wait):
        // slot 0/1 for the per-tile max exchange (by tile parity), 2 at the end
        auto pair_sync = [&](int slot, uint32_t parity) {
            mbar_arrive(&bar_pair[quad][slot]);
            return mbar_wait(&bar_pair[quad][slot], parity);
        };
        float m_used = -INFINITY;
        float l = 0.f;                             // this half's share of the row sum
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            const int k0 = (t_begin + j) * kTcN;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_s_full[sb], (j >> 1) & 1)) ||
                *reinterpret_cast<volatile int*>(&s_fail)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const uint32_t s_col = lane_base + sb * kTcN + half * 64;
            const int kh = k0 + half * 64;          // first key of this half
            const bool full_vis = (!a.causal || k0 + kTcN - 1 <= pos_min) && (k0 + kTcN <= kv_len) &&
                                  (a.window <= 0 || k0 > pos_max - a.window);
            float x[64];
            tc::ld32(s_col, *reinterpret_cast<float(*)[32]>(x));
            tc::ld32(s_col + 32, *reinterpret_cast<float(*)[32]>(x + 32));
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_s_free[sb]);  // S is in registers
            // Row max.  Tiles wholly visible to the CTA (all but the diagonal and
            // the window edge) take the short path: the max of the raw scores,
            // scaled once.  Masked tiles scale and mask every score here, so the
            // exponential pass below reads them ready.
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full_vis) {
#pragma unroll
                for (int e = 0; e < 64; ++e) m4[e & 3] = fmaxf(m4[e & 3], x[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const int key = kh + e;
                    const bool vis = key < kv_len && (!a.causal || key <= pos) &&
                                     (a.window <= 0 || key > pos - a.window);
                    x[e] = vis ? x[e] * scale_log2 : -INFINITY;
                    m4[e & 3] = fmaxf(m4[e & 3], x[e]);
                }
            }
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            if (full_vis) mx *= scale_log2;  // scale_log2 > 0: the max commutes with it
            s_red_max[sb][half][r] = mx;
            if (!__all_sync(0xFFFFFFFFu, pair_sync(sb, (j >> 1) & 1))) {
                ok = false;
                break;
            }
            mx = fmaxf(mx, s_red_max[sb][half ^ 1][r]);
            // lazy rescale: keep a stale max unless the new one exceeds it by 2^8
            const float m_new = fmaxf(m_used, mx);
            const bool need = m_new > m_used + kRescaleThreshold ||
                              (m_used == -INFINITY && m_new != -INFINITY);
            float alpha = 1.f;
            if (need) {
                alpha = m_used == -INFINITY ? 0.f : fast_exp2(m_used - m_new);
                m_used = m_new;
                l *= alpha;
            }
            // keys past kv_len in the last tile: zero their V rows so that a
            // NaN in an unused slot never meets a zero weight in the MMA
            if (k0 + kTcN > kv_len) {
                const int st = j % C::kVStages;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_v[st], (j / C::kVStages) & 1))) {
                    ok = false;
                    break;
                }
                uint8_t* sV = smem + C::kOffV + st * C::kKBytes;
                const int first = max(0, kv_len - k0);
                // 8 warps x 32 lanes zero rows [first, 128) of every half
                for (int row = first + (sm_tid >> 3); row < kTcN; row += 32) {
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        *reinterpret_cast<uint4*>(sV + h * C::kHalfBytes + row * 128 + (sm_tid & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // PV_{j-1} must be done before O is rescaled or P is overwritten
            if (j > 0) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_o_done, (j - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                if (__any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        float v[32];
                        const uint32_t col = lane_base + C::kColO + half * (D / 2) + c * 32;
                        tc::ld32(col, v);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= alpha;
                        tc::st32(col, v);
                    }
                    tc::wait_st();
                }
            }
            // P = 2^(x - m) in fp32 (the row sum l stays exact to fp32), packed
            // to bf16 pairs into the swizzled K-major P tile (this half's keys)
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            // p = 2^(score * scale - mu): one FMA and one exp2 per score on the
            // short path (raw scores), one subtract on the masked path
            const float sc = full_vis ? scale_log2 : 1.f;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {              // 8 chunks of 8 keys
                uint32_t pk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float p0 = fast_exp2(fmaf(x[q8 * 8 + 2 * u], sc, -mu));
                    const float p1 = fast_exp2(fmaf(x[q8 * 8 + 2 * u + 1], sc, -mu));
                    s4[u] += p0 + p1;
                    pk[u] = pack2<false>(p0, p1);
                }
                *reinterpret_cast<uint4*>(sP + half * C::kHalfBytes + sw128(r, q8)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_p_full);
        }
        if (ok && n_tiles > 0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_o_done, (n_tiles - 1) & 1));
            tc::fence_after_sync();
        }
        // every softmax thread reaches this exchange (failure or not; the wait is bounded)
        s_red_sum[half][r] = l;
        if (!__all_sync(0xFFFFFFFFu, pair_sync(2, 0))) ok = false;
        const float l_row = l + s_red_sum[half ^ 1][r];
        if (!ok) {
            if (lane == 0) {
                flag_error(a.err, PKV_DEVERR_TIMEOUT);
                atomicOr(&s_fail, 1);
            }
        } else {
            // epilogue: this half's O columns / l -> bf16; lse by half 0
            const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                                  (static_cast<size_t>(q0 + tok0 + t) * a.hq + kvh * G + r % G) * D +
                                  half * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                float v[32];
                if (n_tiles > 0) {
                    tc::ld32(lane_base + C::kColO + half * (D / 2) + c * 32, v);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.f;
                }
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        *reinterpret_cast<uint4*>(orow + c * 32 + e) =
                            make_uint4(pack2<false>(v[e] * inv, v[e + 1] * inv),
                                       pack2<false>(v[e + 2] * inv, v[e + 3] * inv),
                                       pack2<false>(v[e + 4] * inv, v[e + 5] * inv),
                                       pack2<false>(v[e + 6] * inv, v[e + 7] * inv));
                    }
                }
            }
            if (row_ok && a.lse_out && half == 0)
                a.lse_out[static_cast<size_t>(q0 + tok0 + t) * a.hq + kvh * G + r % G] =
                    l_row > 0.f ? (m_used + __log2f(l_row)) * 0.6931471805599453f : -INFINITY;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
cudaError_t launch_prefill_tc_t(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t stream) {
    using C = TcCfg<D>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    auto kern = prefill_tc_kernel<D>;
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
    return launch_pdl(kern, grid, dim3(kTcThreads), C::kSmemBytes, stream, a, qmap, kmap, vmap);
}

}  // namespace

int prefill_tc_q_tile(int group) { return group >= 1 && group <= kTcM ? kTcM / group : 0; }

cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t stream) {
    return a.d == 64 ? launch_prefill_tc_t<64>(a, qmap, kmap, vmap, stream)
                     : launch_prefill_tc_t<128>(a, qmap, kmap, vmap, stream);
}

}  // namespace pkv
