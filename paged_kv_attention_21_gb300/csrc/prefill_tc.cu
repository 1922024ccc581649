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
// One CTA owns (sequence, KV head, pair of query tiles A and B).  A tile packs
// QT = 128 / G consecutive query tokens x the G heads of one KV group into
// M = 128 rows (row r -> token r / G, head r % G); the two tiles cover 2 QT
// consecutive tokens and share every K/V tile the CTA reads, so each TMA box
// feeds 256 query rows.  Warp roles:
//   warp 0       TMA producer: both Q tiles once (3-D tensor map over q), then
//                K and V tiles of 128 keys (8 blocks) into separate rings
//                (2 stages each; K frees once both S MMAs are done, V once
//                both PV MMAs are done);
//   warp 1       MMA issuer (one thread), per KV tile j in the order
//                S_A(j) | PV_B(j-1) | S_B(j) | PV_A(j), so that the tensor
//                pipe works on one tile while the softmax warps of the other
//                turn its S into P;
//   warps 2..17  softmax, eight warps per Q tile, two threads per row (its
//                TMEM lane; 64 key columns each, row maxima exchanged in
//                shared memory): masked row max, lazy rescale of O only when
//                the max grows by more than 2^8, P = 2^(x - m) (fp32 exp2,
//                packed to bf16) written back into the tile's S columns of
//                TMEM, and the final 1/l normalisation and bf16 store.
// TMEM (512 columns): S_A | S_B | O_A | O_B.  P_X overwrites the first 64
// columns of S_X, so S_X(j+1) is issued only after PV_X(j) is done; the other
// tile's MMA sits between the two in the order above.  Operands: Q, K (K-major, SW128) via
// shared-memory descriptors, P from TMEM, V read MN-major (head_dim
// contiguous), as stored.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTcM = 128;                         // query rows per tile
constexpr int kTcN = 128;                         // keys per KV tile
constexpr int kTcBlocks = kTcN / kBlockSize;      // 8 blocks per KV tile
constexpr int kTcQTiles = 2;                      // query tiles per CTA (A, B)
constexpr int kTcWarps = 2 + 8 * kTcQTiles;       // producer, MMA issuer, 8 softmax warps per tile
constexpr int kTcThreads = kTcWarps * 32;
constexpr float kRescaleThreshold = 8.0f;         // log2 of the largest stale-max factor

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;             // 64-column (128-byte) halves of a row
    static constexpr int kHalfBytes = 128 * 128;       // 128 rows x 128 bytes
    static constexpr int kQBytes = kHalves * kHalfBytes;  // one Q tile
    static constexpr int kKBytes = kHalves * kHalfBytes;  // 128 keys x D (K or V tile)
    static constexpr int kKStages = 2;
    static constexpr int kVStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTcQTiles * kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    static constexpr int kBodyBytes = kOffV + kVStages * kKBytes;
    // at least 120 KB so that one CTA owns an SM (and all 512 TMEM columns)
    static constexpr int kSmemBytes = (kBodyBytes + 1024 > 120 * 1024) ? kBodyBytes + 1024 : 120 * 1024;
    static constexpr uint32_t kTmemCols = 512;            // S_A | S_B | O_A | O_B
    static constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x * kTcN); }
    static constexpr uint32_t col_o(int x) { return static_cast<uint32_t>(kTcQTiles * kTcN + x * D); }
};

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// The KV tiles one query tile needs, as a range [lo, hi) of tile indices.
struct TileSpan {
    int tok0, ntok;      // first token (within the sequence) and token count
    int pos_min, pos_max;
    int lo, hi;          // absolute KV tile indices
};

__device__ __forceinline__ TileSpan tile_span(int tok0, int q_len, int QT, int kv_len, int causal,
                                              int window) {
    TileSpan t;
    t.tok0 = tok0;
    t.ntok = max(0, min(QT, q_len - tok0));
    const int off = kv_len - q_len;
    t.pos_min = off + tok0;
    t.pos_max = off + tok0 + t.ntok - 1;
    const int key_hi = causal ? min(t.pos_max, kv_len - 1) : kv_len - 1;
    const int key_lo = window > 0 ? max(0, t.pos_min - window + 1) : 0;
    if (t.ntok > 0 && key_hi >= key_lo) {
        t.lo = key_lo / kTcN;
        t.hi = key_hi / kTcN + 1;
    } else {
        t.lo = t.hi = 0;
    }
    return t;
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
    __shared__ __align__(8) uint64_t bar_k[C::kKStages];
    __shared__ __align__(8) uint64_t bar_k_empty[C::kKStages];
    __shared__ __align__(8) uint64_t bar_v[C::kVStages];
    __shared__ __align__(8) uint64_t bar_v_empty[C::kVStages];
    __shared__ __align__(8) uint64_t bar_s_full[kTcQTiles];
    __shared__ __align__(8) uint64_t bar_p_full[kTcQTiles];
    __shared__ __align__(8) uint64_t bar_o_done[kTcQTiles];
    __shared__ __align__(8) uint64_t bar_pair[kTcQTiles][4][3];  // per tile and quadrant: parity 0/1, final
    __shared__ __align__(8) uint64_t bar_mma_fin;  // every MMA this CTA issued is complete
    __shared__ __align__(8) uint64_t probe;        // test hook: a barrier nothing arrives on
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    __shared__ float s_red_max[kTcQTiles][2][2][kTcM];  // [tile][parity][column half][row]
    __shared__ float s_red_sum[kTcQTiles][2][kTcM];     // [tile][column half][row]

    pdl_wait();
    pdl_launch_dependents();
    const int kvh = blockIdx.y;
    const int seq = a.ordered ? static_cast<int>(a.seq_order[blockIdx.z]) : static_cast<int>(blockIdx.z);
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
    const int npairs = (ntiles_q + kTcQTiles - 1) / kTcQTiles;
    if (static_cast<int>(blockIdx.x) >= npairs) return;
    const int pr = npairs - 1 - static_cast<int>(blockIdx.x);  // heaviest pairs first
    TileSpan span[kTcQTiles];
#pragma unroll
    for (int x = 0; x < kTcQTiles; ++x)
        span[x] = tile_span((pr * kTcQTiles + x) * QT, q_len, QT, kv_len, a.causal, a.window);
    // the CTA's KV range is the union of the two tiles' ranges; j below counts
    // KV tiles from t_begin, and tile x is active for j in [jlo[x], jhi[x])
    int t_begin = 1 << 30, t_end = 0;
#pragma unroll
    for (int x = 0; x < kTcQTiles; ++x) {
        if (span[x].hi > span[x].lo) {
            t_begin = min(t_begin, span[x].lo);
            t_end = max(t_end, span[x].hi);
        }
    }
    const int n_tiles = t_end > 0 ? t_end - t_begin : 0;
    int jlo[kTcQTiles], jhi[kTcQTiles];
#pragma unroll
    for (int x = 0; x < kTcQTiles; ++x) {
        jlo[x] = span[x].hi > span[x].lo ? span[x].lo - t_begin : 0;
        jhi[x] = span[x].hi > span[x].lo ? span[x].hi - t_begin : 0;
    }
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
        for (int x = 0; x < kTcQTiles; ++x) {
            mbar_init(&bar_s_full[x], 1);
            mbar_init(&bar_p_full[x], 8);
            mbar_init(&bar_o_done[x], 1);
            for (int qd = 0; qd < 4; ++qd)
                for (int i = 0; i < 3; ++i) mbar_init(&bar_pair[x][qd][i], 64);
        }
        mbar_init(&bar_mma_fin, 1);
        if (a.inject_timeout) mbar_init(&probe, 1);
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

    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.mbps;
    // Waits give up at the time limit, or as soon as another warp has given
    // up (s_fail); the drains at the end wait for copies and MMAs in flight
    // regardless of s_fail.
    const volatile int* abort = &s_fail;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int k_issued = 0, v_issued = 0;   // K / V tiles whose loads were issued
        if (n_tiles > 0) {
            if (lane == 0) {
                int nq = 0;
#pragma unroll
                for (int x = 0; x < kTcQTiles; ++x) nq += span[x].ntok > 0 ? 1 : 0;
                mbar_arrive_expect_tx(&bar_q, nq * C::kHalves * 64 * 2 * G * QT);
#pragma unroll
                for (int x = 0; x < kTcQTiles; ++x) {
                    if (span[x].ntok <= 0) continue;
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(smem + C::kOffQ + x * C::kQBytes + h * C::kHalfBytes, &qmap, &bar_q,
                                    h * 64, kvh * G, q0 + span[x].tok0);
                }
            }
            // order of loads: K_0, K_1, V_0, K_2, V_1, ... -- K one tile ahead of V.
            // Block ids: lane l holds block l % 8 of tile l / 8 of a group of four
            // tiles; the next group is read one group ahead, so the table read is
            // never on the load path.  An id is checked when its group comes up.
            const int blk_end = min(nblk_seq, (t_begin + n_tiles) * kTcBlocks);
            auto read_ids = [&](int grp) -> int {
                const int blk = (t_begin + grp * 4) * kTcBlocks + lane;
                return blk < blk_end ? __ldg(bt + blk) : 0;
            };
            auto check_ids = [&](int v) -> int {
                if (v < 0 || v >= a.num_blocks) {
                    flag_error(a.err, PKV_DEVERR_BLOCK_ID);
                    v = 0;
                }
                return v;
            };
            int ids_cur = check_ids(read_ids(0));
            int ids_next = read_ids(1);
            int ids_old = 0;  // the group before ids_cur (V lags K by one tile)
            for (int j = 0; j <= n_tiles; ++j) {
                bool switched = false;
                if (j < n_tiles) {
                    if (j > 0 && (j & 3) == 0) {
                        ids_old = ids_cur;
                        ids_cur = check_ids(ids_next);
                        ids_next = read_ids((j >> 2) + 1);
                        switched = true;
                    }
                    const int blk0 = (t_begin + j) * kTcBlocks;
                    const int st = j % C::kKStages;
                    int ok = 1;
                    if (lane == 0)
                        ok = mbar_wait(&bar_k_empty[st], ((j / C::kKStages) & 1) ^ 1, kWaitLimitNs, abort) ? 1 : 0;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    const int nvalid = min(kTcBlocks, nblk_seq - blk0);
                    uint8_t* sK = smem + C::kOffK + st * C::kKBytes;
                    int ids[kTcBlocks];
#pragma unroll
                    for (int b = 0; b < kTcBlocks; ++b)
                        ids[b] = __shfl_sync(0xFFFFFFFFu, ids_cur, (j & 3) * kTcBlocks + b);
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
                    k_issued = j + 1;
                }
                if (j >= 1) {
                    const int i = j - 1;
                    const int st = i % C::kVStages;
                    int ok = 1;
                    if (lane == 0)
                        ok = mbar_wait(&bar_v_empty[st], ((i / C::kVStages) & 1) ^ 1, kWaitLimitNs, abort) ? 1 : 0;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    const int blk0 = (t_begin + i) * kTcBlocks;
                    const int nvalid = min(kTcBlocks, nblk_seq - blk0);
                    uint8_t* sV = smem + C::kOffV + st * C::kKBytes;
                    const int src = switched ? ids_old : ids_cur;
                    int ids[kTcBlocks];
#pragma unroll
                    for (int b = 0; b < kTcBlocks; ++b)
                        ids[b] = __shfl_sync(0xFFFFFFFFu, src, (i & 3) * kTcBlocks + b);
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
                    v_issued = i + 1;
                }
            }
            // drain: the last load issued into each stage (and Q) has landed
            // before this CTA may exit -- immediate unless a wait gave up
            if (lane == 0) {
                (void)mbar_wait(&bar_q, 0);
                for (int j = max(0, k_issued - C::kKStages); j < k_issued; ++j)
                    (void)mbar_wait(&bar_k[j % C::kKStages], (j / C::kKStages) & 1);
                for (int i = max(0, v_issued - C::kVStages); i < v_issued; ++i)
                    (void)mbar_wait(&bar_v[i % C::kVStages], (i / C::kVStages) & 1);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTcM, kTcN, false, false);
        constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTcM, D, false, true);
        bool ok = n_tiles > 0 ? mbar_wait(&bar_q, 0, kWaitLimitNs, abort) : true;
        ok = __all_sync(0xFFFFFFFFu, ok);
        auto active = [&](int x, int j) { return j >= jlo[x] && j < jhi[x]; };
        // S_x(j) = Q_x K_j^T once PV_x(j-1) is done (it reads P_x(j-1) from the
        // columns S_x(j) overwrites).  A 128-key S is one N = 128 MMA per k-step:
        // two N = 64 halves cost as much tensor time each as one N = 128.
        auto issue_s = [&](int x, int j) -> bool {
            const int ks = j % C::kKStages;
            const uint8_t* sQ = smem + C::kOffQ + x * C::kQBytes;
            const uint8_t* sK = smem + C::kOffK + ks * C::kKBytes;
            if (j > jlo[x]) {
                const bool r = mbar_wait(&bar_o_done[x], (j - 1 - jlo[x]) & 1, kWaitLimitNs, abort);
                if (!__all_sync(0xFFFFFFFFu, r)) return false;
                tc::fence_after_sync();
            }
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int h = kk >> 2;
                    const uint32_t ko = (kk & 3) * 32;
                    const uint64_t ad = tc::smem_desc(smem_u32(sQ + h * C::kHalfBytes) + ko, 16, 1024);
                    const uint64_t bd = tc::smem_desc(smem_u32(sK + h * C::kHalfBytes) + ko, 16, 1024);
                    tc::mma_bf16(tmem + C::col_s(x), ad, bd, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bar_s_full[x]);
            }
            __syncwarp();
            return true;
        };
        // O_x += P_x(j) V_j with P read from the first 64 columns of S_x
        auto issue_pv = [&](int x, int j) -> bool {
            const int vs = j % C::kVStages;
            const bool r1 = mbar_wait(&bar_p_full[x], (j - jlo[x]) & 1, kWaitLimitNs, abort);
            const bool r2 = r1 && mbar_wait(&bar_v[vs], (j / C::kVStages) & 1, kWaitLimitNs, abort);
            if (!__all_sync(0xFFFFFFFFu, r1 && r2)) return false;
            tc::fence_after_sync();
            if (lane == 0) {
                const uint8_t* sV = smem + C::kOffV + vs * C::kKBytes;
#pragma unroll
                for (int kk = 0; kk < kTcN / 16; ++kk) {
                    // P column group kk holds keys 64 c + 32 h + 16 s with h = kk / 4,
                    // c = (kk / 2) % 2, s = kk % 2 (the softmax layout below).
                    // V, MN-major: 16 keys per k-step = 2 groups of 8 rows (SBO 1024);
                    // the two 64-column halves of head_dim are C::kHalfBytes apart (LBO)
                    const int vrow = 64 * ((kk >> 1) & 1) + 32 * (kk >> 2) + 16 * (kk & 1);
                    const uint64_t bd = tc::smem_desc(smem_u32(sV) + vrow * 128, C::kHalfBytes, 1024);
                    tc::mma_bf16_tmem_a(tmem + C::col_o(x), tmem + C::col_s(x) + kk * 8, bd, kIdescPV,
                                        (j > jlo[x] || kk > 0) ? 1u : 0u);
                }
                tc::commit(&bar_o_done[x]);
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; ok && j <= n_tiles; ++j) {
            if (j < n_tiles) {
                const int ks = j % C::kKStages;
                const bool inject = a.inject_timeout != 0 && j == 0 && is_first_cta();
                const bool r = inject ? mbar_wait(&probe, 0, 1000ull * a.inject_limit_us, abort)
                                      : mbar_wait(&bar_k[ks], (j / C::kKStages) & 1, kWaitLimitNs, abort);
                if (!__all_sync(0xFFFFFFFFu, r) || *reinterpret_cast<volatile int*>(&s_fail)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                if (active(0, j) && !issue_s(0, j)) { ok = false; break; }
                if (!active(1, j)) {
                    if (lane == 0) tc::commit(&bar_k_empty[ks]);
                    __syncwarp();
                }
            }
            if (j >= 1 && active(1, j - 1)) {
                if (!issue_pv(1, j - 1)) { ok = false; break; }
                if (lane == 0) tc::commit(&bar_v_empty[(j - 1) % C::kVStages]);
                __syncwarp();
            }
            if (j < n_tiles) {
                if (active(1, j)) {
                    if (!issue_s(1, j)) { ok = false; break; }
                    if (lane == 0) tc::commit(&bar_k_empty[j % C::kKStages]);  // K_j no longer needed
                    __syncwarp();
                }
                if (active(0, j)) {
                    if (!issue_pv(0, j)) { ok = false; break; }
                    if (!active(1, j)) {
                        if (lane == 0) tc::commit(&bar_v_empty[j % C::kVStages]);
                        __syncwarp();
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            atomicOr(&s_fail, 1);
        }
        // drain: every MMA this thread issued is complete before TMEM is
        // freed and the CTA exits (immediate unless a wait gave up)
        if (lane == 0) tc::commit(&bar_mma_fin);
        __syncwarp();
        (void)mbar_wait(&bar_mma_fin, 0);
        tc::fence_after_sync();
    } else {
        // -------------------------------------------------------------- softmax
        // Warp w (2..17) serves query tile x = (w - 2) / 8 and reads TMEM lane
        // quadrant w % 4; two warps share each quadrant.  Half h = ((w - 2) / 4) % 2
        // owns the S columns 64 c + 32 h + [0, 32) for c = 0, 1 (keys k0 + the
        // same offsets) and O columns [h D/2, (h+1) D/2).  The pair exchanges row
        // maxima through shared memory; row sums stay per half.  Scores are
        // streamed from TMEM twice (max, then exponentials): P for chunk c goes
        // to columns 32 h + 16 c + [0, 16), which this half has already read, so
        // P_x fills columns [0, 64) of S_x.
        const int sw = warp - 2;
        const int x = sw >> 3;                     // query tile
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int half = (sw >> 2) & 1;            // key / O column half
        const int r = quad * 32 + lane;            // the row this thread owns
        const int t = r / G;
        const TileSpan sp = x ? span[1] : span[0];
        const bool row_ok = r < QT * G && t < sp.ntok;
        const int pos = sp.pos_min + t;
        const int j0 = x ? jlo[1] : jlo[0];
        const int nx = x ? jhi[1] - jlo[1] : jhi[0] - jlo[0];
        const float scale_log2 = a.sm_scale * 1.4426950408889634f * (a.k_scale ? a.k_scale[kvh] : 1.f);
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t s_base = lane_base + C::col_s(x);
        const int grp_tid = (sw & 7) * 32 + lane;  // 0..255 within the tile's softmax group
        // the two warps of this quadrant meet on an mbarrier (bounded wait):
        // slot 0/1 for the per-tile max exchange (by tile parity), 2 at the end
        auto pair_sync = [&](int slot, uint32_t parity) {
            mbar_arrive(&bar_pair[x][quad][slot]);
            return mbar_wait(&bar_pair[x][quad][slot], parity, kWaitLimitNs, abort);
        };
        float m_used = -INFINITY;
        float l = 0.f;                             // this half's share of the row sum
        bool ok = true;
        for (int i = 0; i < nx; ++i) {
            const int j = j0 + i;
            const int k0 = (t_begin + j) * kTcN;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_s_full[x], i & 1, kWaitLimitNs, abort)) ||
                *reinterpret_cast<volatile int*>(&s_fail)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const bool full_vis = (!a.causal || k0 + kTcN - 1 <= sp.pos_min) && (k0 + kTcN <= kv_len) &&
                                  (a.window <= 0 || k0 > sp.pos_max - a.window);
            // Row max.  Tiles wholly visible to the CTA (all but the diagonal and
            // the window edge) take the max of the raw scores, scaled once;
            // masked tiles scale and mask every score.
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float xs[32];
                tc::ld32(s_base + 64 * c + 32 * half, xs);
                tc::wait_ld();
                if (full_vis) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], xs[e]);
                } else {
                    const int kb = k0 + 64 * c + 32 * half;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = kb + e;
                        const bool vis = key < kv_len && (!a.causal || key <= pos) &&
                                         (a.window <= 0 || key > pos - a.window);
                        m4[e & 3] = fmaxf(m4[e & 3], vis ? xs[e] * scale_log2 : -INFINITY);
                    }
                }
            }
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            if (full_vis) mx *= scale_log2;  // scale_log2 > 0: the max commutes with it
            s_red_max[x][i & 1][half][r] = mx;
            if (!__all_sync(0xFFFFFFFFu, pair_sync(i & 1, (i >> 1) & 1))) {
                ok = false;
                break;
            }
            mx = fmaxf(mx, s_red_max[x][i & 1][half ^ 1][r]);
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
            // NaN in an unused slot never meets a zero weight in the MMA.  The
            // tile whose PV reads V_j first does it (A when it uses V_j).
            const bool zero_v = k0 + kTcN > kv_len && (x == 0 || j < jlo[0] || j >= jhi[0]);
            if (zero_v) {
                const int st = j % C::kVStages;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar_v[st], (j / C::kVStages) & 1, kWaitLimitNs, abort))) {
                    ok = false;
                    break;
                }
                uint8_t* sV = smem + C::kOffV + st * C::kKBytes;
                const int first = max(0, kv_len - k0);
                // 8 warps x 32 lanes zero rows [first, 128) of every half
                for (int row = first + (grp_tid >> 3); row < kTcN; row += 32) {
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        *reinterpret_cast<uint4*>(sV + h * C::kHalfBytes + row * 128 + (grp_tid & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
            }
            // P = 2^(x - m) in fp32 (the row sum l stays exact to fp32), packed to
            // bf16 pairs (the lower key in the low half)
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float xs[32];
                tc::ld32(s_base + 64 * c + 32 * half, xs);
                tc::wait_ld();
                uint32_t pk[16];
                if (full_vis) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float p0 = fast_exp2(fmaf(xs[2 * u], scale_log2, -mu));
                        const float p1 = fast_exp2(fmaf(xs[2 * u + 1], scale_log2, -mu));
                        s4[u & 3] += p0 + p1;
                        pk[u] = pack2<false>(p0, p1);
                    }
                } else {
                    const int kb = k0 + 64 * c + 32 * half;
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        float pp[2];
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            const int key = kb + 2 * u + v;
                            const bool vis = key < kv_len && (!a.causal || key <= pos) &&
                                             (a.window <= 0 || key > pos - a.window);
                            pp[v] = vis ? fast_exp2(fmaf(xs[2 * u + v], scale_log2, -mu)) : 0.f;
                        }
                        s4[u & 3] += pp[0] + pp[1];
                        pk[u] = pack2<false>(pp[0], pp[1]);
                    }
                }
                tc::st16u(s_base + 32 * half + 16 * c, pk);
            }
            l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
            // PV_x(j-1) is done (S_x(j) was issued after it), so O may be rescaled
            if (i > 0 && __any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    float v[32];
                    const uint32_t col = lane_base + C::col_o(x) + half * (D / 2) + c * 32;
                    tc::ld32(col, v);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= alpha;
                    tc::st32(col, v);
                }
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_p_full[x]);
        }
        if (ok && nx > 0) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_o_done[x], (nx - 1) & 1, kWaitLimitNs, abort));
            tc::fence_after_sync();
        }
        // every softmax thread reaches this exchange (failure or not; the wait is bounded)
        s_red_sum[x][half][r] = l;
        if (!__all_sync(0xFFFFFFFFu, pair_sync(2, 0))) ok = false;
        const float l_row = l + s_red_sum[x][half ^ 1][r];
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            atomicOr(&s_fail, 1);
        }
        if (sp.ntok > 0) {
            // epilogue: this half's O columns / l -> bf16 (or fp32); lse by half 0.
            // A tile that gave up writes o = 0 and lse = -inf.
            const float inv = ok && l_row > 0.f ? (a.v_scale ? a.v_scale[kvh] : 1.f) / l_row : 0.f;
            const size_t orow0 = (static_cast<size_t>(q0 + sp.tok0 + t) * a.hq + kvh * G + r % G) * D + half * (D / 2);
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + orow0;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                float v[32];
                if (nx > 0 && ok) {
                    tc::ld32(lane_base + C::col_o(x) + half * (D / 2) + c * 32, v);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.f;
                }
                if (row_ok && a.out_f32) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(a.out_f32 + orow0 + c * 32 + e) =
                            make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
                } else if (row_ok) {
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
                a.lse_out[static_cast<size_t>(q0 + sp.tok0 + t) * a.hq + kvh * G + r % G] =
                    ok && l_row > 0.f ? (m_used + __log2f(l_row)) * 0.6931471805599453f : -INFINITY;
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
    dim3 grid((a.max_qtiles + kTcQTiles - 1) / kTcQTiles, a.hkv, a.num_seqs);
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
