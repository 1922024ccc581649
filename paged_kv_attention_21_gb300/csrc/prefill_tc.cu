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
//                the K tiles of 128 keys (8 blocks, one 4 KiB box each) into
//                a 2-stage ring that frees once both S MMAs are done;
//   warp 10      TMA producer of the V tiles, likewise (frees once both PV
//                MMAs are done);
//   warp 1       MMA issuer (one thread), per KV tile j in the order
//                S_A(j) | PV_B(j-1) | S_B(j) | PV_A(j), so that the tensor
//                pipe works on one tile while the softmax warps of the other
//                turn its S into P;
//   warps 2..9   softmax, four warps per Q tile, one thread per row (its TMEM
//                lane, all 128 key columns): masked row max, lazy rescale of
//                O only when the max grows by more than 2^8, P = 2^(x - m)
//                (fp32 exp2, packed to bf16) written back into the tile's S
//                columns of TMEM, and the final 1/l normalisation and store.
// TMEM (512 columns): S_A | S_B | O_A | O_B.  P_X overwrites the first 64
// columns of S_X, and S_X(j+1) (issued after PV_X(j) by the same thread)
// overwrites them again: the tensor pipe runs one CTA's MMAs in issue order,
// so PV_X(j) has read P_X(j) before S_X(j+1) writes, and S_X(j+1) complete
// implies PV_X(j) complete.  The PTX ISA promises issue order only for MMAs
// into the same accumulator; this kernel relies on it across S and O, as
// FlashAttention-4's Blackwell forward kernel does, and the parity tests
// would show a violation.  Waiting for PV_X(j) before issuing S_X(j+1)
// instead measured 8 % slower.  Operands: Q, K (K-major, SW128) via
// shared-memory descriptors, P from TMEM, V read MN-major (head_dim
// contiguous), as stored.
//
// e4m3 pools (kFp8; InferX, "The kernels underneath": FP8 KV cache): the
// producers TMA each (block, head) box of codes into one of eight one-block
// slots and convert it exactly to f16, in the layout above, into the ring
// stage; the softmax warps turn Q into f16 in place, P is packed as f16, and
// the MMAs run f16 x f16 -> fp32 (one operand type per MMA).  k_scale folds
// into the logit scale and v_scale into the final normalisation.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTcM = 128;                         // query rows per tile
constexpr int kTcN = 128;                         // keys per KV tile
constexpr int kTcBlocks = kTcN / kBlockSize;      // 8 blocks per KV tile
constexpr int kTcQTiles = 2;                      // query tiles per CTA (A, B)
constexpr int kTcSmWarps = 4;                     // softmax warps per query tile: one thread per row
constexpr int kTcVWarp = 2 + kTcSmWarps * kTcQTiles;  // the V producer, after the softmax warps
constexpr int kTcWarps = kTcVWarp + 1;  // K producer, MMA issuer, softmax warps, V producer
constexpr int kTcThreads = kTcWarps * 32;
constexpr float kRescaleThreshold = 8.0f;         // log2 of the largest stale-max factor

template <int D, bool kFp8 = false>
struct TcCfg {
    static constexpr int kHalves = D / 64;             // 64-column (128-byte) halves of a row
    static constexpr int kHalfBytes = 128 * 128;       // 128 rows x 128 bytes
    static constexpr int kQBytes = kHalves * kHalfBytes;  // one Q tile
    static constexpr int kKBytes = kHalves * kHalfBytes;  // 128 keys x D (K or V tile)
    static constexpr int kBlkBytes = kBlockSize * D * 2;   // one (block, head) tile: one TMA box
    static constexpr int kGrpBytes = kHalves * 1024;       // between 8-row groups of a K / V tile
    // a third K stage (224 KiB in all at D = 128) measured no faster: the
    // per-tile chain S -> softmax -> PV of each query tile sets the pace
    static constexpr int kKStages = 2;
    static constexpr int kVStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTcQTiles * kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    // e4m3 pools: eight one-block slots of codes for K and eight for V (one
    // (block, head) box each, [16 rows][D bytes]); a producer converts slot b
    // into block b of its f16 ring stage, then refills the slot with block b
    // of the next tile, so seven loads stay in flight behind each conversion
    static constexpr int kStgBlkBytes = kBlockSize * D;    // one (block, head) box of codes
    static constexpr int kStgBytes = kFp8 ? kTcBlocks * kStgBlkBytes : 0;
    static constexpr int kOffSK = kOffV + kVStages * kKBytes;
    static constexpr int kOffSV = kOffSK + kStgBytes;
    static constexpr int kBodyBytes = kOffSV + kStgBytes;
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

// One (block, head) box of e4m3 codes ([16 rows][D bytes], as the unswizzled
// TMA box writes it) -> that block's f16 rows in a ring stage, in the layout
// the tile-group box writes for 16-bit pools: [8-row group][64-column slice]
// [8 rows][128 B, 16-byte chunks swizzled by the row].  Lane l converts the
// 8 codes of chunk l % (D/8) in rows l / (D/8), + 32 / (D/8), ...: a row's
// codes are read by consecutive lanes and its chunks land in distinct banks.
// e4m3 -> f16 is exact.
template <int D>
__device__ __forceinline__ void convert_e4m3_block(const uint8_t* codes, uint8_t* dst, int lane) {
    using C = TcCfg<D, true>;
    constexpr int kCh = D / 8;                    // 16-byte f16 chunks of a key row
    constexpr int kRowsPerPass = 32 / kCh;
    constexpr int kPasses = kBlockSize / kRowsPerPass;
    const int cg = lane % kCh;
    const int r0 = lane / kCh;
    // all of the lane's codes first: the loads overlap, and no store of the
    // stage has to be ordered before a load of the slot
    uint2 w[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i)
        w[i] = *reinterpret_cast<const uint2*>(codes + (r0 + i * kRowsPerPass) * D + cg * 8);
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const int t = r0 + i * kRowsPerPass;
        uint4 o;
        e4m3x4_to_f16x4(w[i].x, o.x, o.y);
        e4m3x4_to_f16x4(w[i].y, o.z, o.w);
        const int r = t & 7;
        *reinterpret_cast<uint4*>(dst + (t >> 3) * C::kGrpBytes + (cg >> 3) * 1024 + r * 128 +
                                  (((cg & 7) ^ r) << 4)) = o;
    }
}

template <int D, bool kFp8>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
    using C = TcCfg<D, kFp8>;
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
    __shared__ __align__(8) uint64_t bar_mma_fin;  // every MMA this CTA issued is complete
    __shared__ __align__(8) uint64_t bar_stg[2][kTcBlocks];  // e4m3: K / V code slot b has landed
    __shared__ __align__(8) uint64_t bar_qc;       // e4m3: the softmax warps turned Q into f16
    __shared__ __align__(8) uint64_t probe;        // test hook: a barrier nothing arrives on
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;

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
            mbar_init(&bar_p_full[x], kTcSmWarps);
            mbar_init(&bar_o_done[x], 1);
        }
        mbar_init(&bar_mma_fin, 1);
        if constexpr (kFp8) {
            for (int b = 0; b < kTcBlocks; ++b) {
                mbar_init(&bar_stg[0][b], 1);
                mbar_init(&bar_stg[1][b], 1);
            }
            mbar_init(&bar_qc, kTcSmWarps * kTcQTiles);
        }
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

    if (warp == 0 || warp == kTcVWarp) {
        // ----------------------------------------------------------- producers
        // Warp 0 loads Q and the K tiles, warp kTcVWarp the V tiles: one
        // thread issues a TMA copy only every ~200 cycles, so the two rings
        // are fed in parallel.  Each (block, head) tile is one 5-D box, laid
        // out [row group][64-column slice][8 rows][128 B] (see the tensor map).
        const bool is_v = warp == kTcVWarp;
        int issued = 0;   // tiles whose loads were issued
        if (n_tiles > 0) {
            if (!is_v && lane == 0) {
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
            const CUtensorMap* map = is_v ? &vmap : &kmap;
            if constexpr (kFp8) {
                // e4m3 pools: block b of every tile passes through code slot b.
                // Lane b issues slot b's loads; the whole warp converts a
                // landed slot into the tile's f16 ring stage, and lane b then
                // loads block b of the next tile into it.
                uint8_t* stg = smem + (is_v ? C::kOffSV : C::kOffSK);
                uint64_t* sbar = bar_stg[is_v ? 1 : 0];
                const int nst = is_v ? C::kVStages : C::kKStages;
                int mylast = -1;   // lane b < 8: the last tile loaded into slot b
                {   // tile 0: lane b < 8 loads its block b
                    const int nv = min(kTcBlocks, nblk_seq - t_begin * kTcBlocks);
                    const int id = __shfl_sync(0xFFFFFFFFu, ids_cur, lane & (kTcBlocks - 1));
                    if (lane < nv) {
                        mbar_arrive_expect_tx(&sbar[lane], C::kStgBlkBytes);
                        tma_load_4d(stg + lane * C::kStgBlkBytes, map, &sbar[lane], 0, 0, kvh, id);
                        mylast = 0;
                    }
                }
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j % nst;
                    uint64_t* full = is_v ? &bar_v[st] : &bar_k[st];
                    uint64_t* empty = is_v ? &bar_v_empty[st] : &bar_k_empty[st];
                    bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(empty, ((j / nst) & 1) ^ 1, kWaitLimitNs, abort));
                    const int nvalid = min(kTcBlocks, nblk_seq - (t_begin + j) * kTcBlocks);
                    const bool more = j + 1 < n_tiles;
                    // rotate the block ids before the next tile's first load
                    int id_next = 0, nv_next = 0;
                    if (more) {
                        if (((j + 1) & 3) == 0) {
                            ids_cur = check_ids(ids_next);
                            ids_next = read_ids(((j + 1) >> 2) + 1);
                        }
                        nv_next = min(kTcBlocks, nblk_seq - (t_begin + j + 1) * kTcBlocks);
                        id_next = __shfl_sync(0xFFFFFFFFu, ids_cur,
                                              ((j + 1) & 3) * kTcBlocks + (lane & (kTcBlocks - 1)));
                    }
                    uint8_t* dst = smem + (is_v ? C::kOffV : C::kOffK) + st * C::kKBytes;
                    for (int b = 0; ok && b < nvalid; ++b) {
                        // every lane reads the codes and writes the stage: all wait
                        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sbar[b], j & 1, kWaitLimitNs, abort));
                        if (!ok) break;
                        convert_e4m3_block<D>(stg + b * C::kStgBlkBytes, dst + b * C::kBlkBytes, lane);
                        // the slot's codes are in registers (the stores depend
                        // on them): the next copy into it may start
                        __syncwarp();
                        if (more && lane == b && b < nv_next) {
                            mbar_arrive_expect_tx(&sbar[b], C::kStgBlkBytes);
                            tma_load_4d(stg + b * C::kStgBlkBytes, map, &sbar[b], 0, 0, kvh, id_next);
                            mylast = j + 1;
                        }
                    }
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    // (only the last tile may have fewer than 8 blocks, so every
                    // slot the next tile needs was refilled above)
                    fence_proxy_async_smem();   // the stage's generic writes -> before the MMAs read it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full);
                }
                // drain: every code load issued (and Q) has landed
                if (lane < kTcBlocks && mylast >= 0) (void)mbar_wait(&sbar[lane], mylast & 1);
                if (lane == 0 && !is_v) (void)mbar_wait(&bar_q, 0);
                __syncwarp();
            } else {
                for (int j = 0; j < n_tiles; ++j) {
                    if (j > 0 && (j & 3) == 0) {
                        ids_cur = check_ids(ids_next);
                        ids_next = read_ids((j >> 2) + 1);
                    }
                    const int blk0 = (t_begin + j) * kTcBlocks;
                    const int nst = is_v ? C::kVStages : C::kKStages;
                    const int st = j % nst;
                    uint64_t* full = is_v ? &bar_v[st] : &bar_k[st];
                    uint64_t* empty = is_v ? &bar_v_empty[st] : &bar_k_empty[st];
                    int ok = 1;
                    if (lane == 0) ok = mbar_wait(empty, ((j / nst) & 1) ^ 1, kWaitLimitNs, abort) ? 1 : 0;
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok || *reinterpret_cast<volatile int*>(&s_fail)) {
                        if (lane == 0) atomicOr(&s_fail, 1);
                        break;
                    }
                    const int nvalid = min(kTcBlocks, nblk_seq - blk0);
                    uint8_t* dst = smem + (is_v ? C::kOffV : C::kOffK) + st * C::kKBytes;
                    // lane b < 8 holds block b of this tile
                    const int id = __shfl_sync(0xFFFFFFFFu, ids_cur, (j & 3) * kTcBlocks + (lane & (kTcBlocks - 1)));
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(full, nvalid * C::kBlkBytes);
                    }
                    __syncwarp();
                    // every block's copy is issued by its own lane, in one instruction
                    if (lane < nvalid) tma_load_5d(dst + lane * C::kBlkBytes, map, full, 0, 0, 0, 0, id * a.hkv + kvh);
                    issued = j + 1;
                }
                // drain: the last load issued into each stage (and Q) has landed
                // before this CTA may exit -- immediate unless a wait gave up
                if (lane == 0) {
                    if (!is_v) (void)mbar_wait(&bar_q, 0);
                    const int nst = is_v ? C::kVStages : C::kKStages;
                    for (int j = max(0, issued - nst); j < issued; ++j)
                        (void)mbar_wait(is_v ? &bar_v[j % nst] : &bar_k[j % nst], (j / nst) & 1);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        // e4m3 pools: Q, K, V and P are all f16 (one operand type per MMA)
        constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTcM, kTcN, false, false, kFp8);
        constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTcM, D, false, true, kFp8);
        bool ok = n_tiles > 0 ? mbar_wait(kFp8 ? &bar_qc : &bar_q, 0, kWaitLimitNs, abort) : true;
        ok = __all_sync(0xFFFFFFFFu, ok);
        auto active = [&](int x, int j) { return j >= jlo[x] && j < jhi[x]; };
        // S_x(j) = Q_x K_j^T, issued right behind PV_x(j-1): the MMAs run in
        // issue order, so PV_x(j-1) reads P_x(j-1) before S_x(j) overwrites it.
        // A 128-key S is one N = 128 MMA per k-step: two N = 64 halves cost as
        // much tensor time each as one N = 128.
        auto issue_s = [&](int x, int j) -> bool {
            const int ks = j % C::kKStages;
            const uint8_t* sQ = smem + C::kOffQ + x * C::kQBytes;
            const uint8_t* sK = smem + C::kOffK + ks * C::kKBytes;
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int h = kk >> 2;
                    const uint32_t ko = (kk & 3) * 32;
                    const uint64_t ad = tc::smem_desc(smem_u32(sQ + h * C::kHalfBytes) + ko, 16, 1024);
                    // K: slice h of every 8-row group, groups C::kGrpBytes apart
                    const uint64_t bd = tc::smem_desc(smem_u32(sK + h * 1024) + ko, 16, C::kGrpBytes);
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
                    // P columns 8 kk .. 8 kk + 7 hold keys 16 kk .. 16 kk + 15 (two
                    // bf16 per column, the lower key in the low half): block kk of
                    // the tile.  V, MN-major: its 2 groups of 8 rows C::kGrpBytes
                    // apart (SBO); the 64-column slices of head_dim 1024 B apart (LBO)
                    const uint64_t bd = tc::smem_desc(smem_u32(sV) + kk * C::kBlkBytes, 1024, C::kGrpBytes);
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
        // Warp w (2..9) serves query tile x = (w - 2) / 4 and reads TMEM lane
        // quadrant w % 4: each thread owns one row (its TMEM lane) and all 128
        // key columns of a tile, so the row max and sum need no exchange.
        // Per KV tile: load the 128 scores, take the masked row max, lazily
        // rescale (only when the max grows by more than 2^8), form P = 2^(x - m)
        // in fp32 (packed f32x2 arithmetic, ex2 on the MUFU), accumulate the row
        // sum, and write P as bf16 pairs over columns [0, 64) of the tile's S.
        const int sw = warp - 2;
        const int x = sw / kTcSmWarps;             // query tile
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
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
        const int grp_tid = (sw % kTcSmWarps) * 32 + lane;  // 0..127 within the tile's softmax group
        bool ok = true;
        if constexpr (kFp8) {
            // e4m3 pools run f16 MMAs: each tile's softmax group turns its Q
            // tile (bf16 as loaded) into f16 in place before the first S
            if (n_tiles > 0) {
                if (sp.ntok > 0) {
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bar_q, 0, kWaitLimitNs, abort));
                    if (ok) {
                        uint4* qt = reinterpret_cast<uint4*>(smem + C::kOffQ + x * C::kQBytes);
                        for (int i = grp_tid; i < C::kQBytes / 16; i += kTcSmWarps * 32) {
                            uint4 v = qt[i];
                            v.x = pack2<true>(bf16_lo(v.x), bf16_hi(v.x));
                            v.y = pack2<true>(bf16_lo(v.y), bf16_hi(v.y));
                            v.z = pack2<true>(bf16_lo(v.z), bf16_hi(v.z));
                            v.w = pack2<true>(bf16_lo(v.w), bf16_hi(v.w));
                            qt[i] = v;
                        }
                        fence_proxy_async_smem();
                    } else if (lane == 0) {
                        atomicOr(&s_fail, 1);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_qc);
            }
        }
        float m_used = -INFINITY;
        float l = 0.f;                             // the row sum
        for (int i = 0; ok && i < nx; ++i) {
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
            float sv[kTcN];
#pragma unroll
            for (int c = 0; c < kTcN / 32; ++c)
                tc::ld32(s_base + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
            tc::wait_ld();
            // Row max.  Tiles wholly visible to the row (all but the diagonal
            // and the window edge) take the max of the raw scores, scaled once;
            // the others scale and mask every score (masked scores become -inf).
            float mx;
            if (full_vis) {
                float m8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
                for (int e = 8; e < kTcN; e += 16) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) m8[u] = fmax3(m8[u], sv[e + u], sv[e + 8 + u]);
                }
                mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                mx *= scale_log2;  // scale_log2 > 0: the max commutes with it
            } else {
                // the row sees keys [key_lo, key_hi]: one unsigned compare per score
                const int key_hi = a.causal ? min(pos, kv_len - 1) : kv_len - 1;
                const int key_lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
                const uint32_t cnt = key_hi >= key_lo ? static_cast<uint32_t>(key_hi + 1 - key_lo) : 0u;
                const int base = k0 - key_lo;
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kTcN; ++e) {
                    const bool vis = static_cast<uint32_t>(base + e) < cnt;
                    sv[e] = vis ? sv[e] * scale_log2 : -INFINITY;
                    m4[e & 3] = fmaxf(m4[e & 3], sv[e]);
                }
                mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
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
                // 4 warps x 32 lanes zero key rows [first, 128), every slice (row t:
                // block t / 16, group (t / 8) % 2, row t % 8 of that group)
                for (int row = first + (grp_tid >> 3); row < kTcN; row += 16) {
                    uint8_t* rp = sV + (row >> 4) * C::kBlkBytes + ((row >> 3) & 1) * C::kGrpBytes + (row & 7) * 128 +
                                  (grp_tid & 7) * 16;
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        *reinterpret_cast<uint4*>(rp + h * 1024) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
            }
            // P = 2^(x - m) in fp32 (the row sum stays exact to fp32), packed to
            // bf16 pairs (the lower key in the low half): keys 32 c .. 32 c + 31
            // go to P columns 16 c .. 16 c + 15
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            const uint64_t scl = pack_f32x2(full_vis ? scale_log2 : 1.f, full_vis ? scale_log2 : 1.f);
            const uint64_t neg = pack_f32x2(-mu, -mu);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < kTcN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const uint64_t xv = fma_f32x2(pack_f32x2(sv[32 * c + 2 * u], sv[32 * c + 2 * u + 1]), scl, neg);
                    float x0, x1;
                    unpack_f32x2(xv, x0, x1);
                    const float p0 = fast_exp2(x0);
                    const float p1 = fast_exp2(x1);
                    const uint64_t pp = pack_f32x2(p0, p1);
                    acc[u & 3] = add_f32x2(acc[u & 3], pp);
                    pk[u] = pack2<kFp8>(p0, p1);
                }
                tc::st16u(s_base + 16 * c, pk);
            }
            {
                float a0, a1, b0, b1, c0, c1, d0, d1;
                unpack_f32x2(add_f32x2(acc[0], acc[1]), a0, a1);
                unpack_f32x2(add_f32x2(acc[2], acc[3]), b0, b1);
                (void)c0; (void)c1; (void)d0; (void)d1;
                l += (a0 + a1) + (b0 + b1);
            }
            // PV_x(j-1) is done (S_x(j), issued after it, is done), so O may be rescaled
            if (i > 0 && __any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    const uint32_t col = lane_base + C::col_o(x) + c * 32;
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
        if (!ok && lane == 0) {
            flag_error(a.err, PKV_DEVERR_TIMEOUT);
            atomicOr(&s_fail, 1);
        }
        if (sp.ntok > 0) {
            // epilogue: the row's O / l -> bf16 (or fp32), and its lse.  A tile
            // that gave up writes o = 0 and lse = -inf.
            const float inv = ok && l > 0.f ? (a.v_scale ? a.v_scale[kvh] : 1.f) / l : 0.f;
            const size_t orow0 = (static_cast<size_t>(q0 + sp.tok0 + t) * a.hq + kvh * G + r % G) * D;
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + orow0;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                if (nx > 0 && ok) {
                    tc::ld32(lane_base + C::col_o(x) + c * 32, v);
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
            if (row_ok && a.lse_out)
                a.lse_out[static_cast<size_t>(q0 + sp.tok0 + t) * a.hq + kvh * G + r % G] =
                    ok && l > 0.f ? (m_used + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool kFp8>
cudaError_t launch_prefill_tc_t(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t stream) {
    using C = TcCfg<D, kFp8>;
    static_assert(C::kSmemBytes <= 227 * 1024, "shared memory budget");
    auto kern = prefill_tc_kernel<D, kFp8>;
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
    if (a.fp8)
        return a.d == 64 ? launch_prefill_tc_t<64, true>(a, qmap, kmap, vmap, stream)
                         : launch_prefill_tc_t<128, true>(a, qmap, kmap, vmap, stream);
    return a.d == 64 ? launch_prefill_tc_t<64, false>(a, qmap, kmap, vmap, stream)
                     : launch_prefill_tc_t<128, false>(a, qmap, kmap, vmap, stream);
}

}  // namespace pkv
