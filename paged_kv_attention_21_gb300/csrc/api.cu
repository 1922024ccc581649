// api.cu -- the C ABI of libpkv: argument validation, split planning,
// tensor-map descriptors, launches and error reporting.  Everything the
// path computes runs in the kernels of decode.cu, prefill_tc.cu and
// append_gather_merge.cu; this file only decides and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <utility>
#include <vector>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/pkv.h"
#include "internal.h"

namespace pkv {
int decode_smem_bytes(int d, int fp8);
}

// One device error word per device (every GPU that loads the library holds
// its own copy).  Kernels get its address as an argument.
__device__ uint32_t g_pkv_device_error;

namespace {

thread_local char g_last_error[512] = "";

// Test hook (pkv_test_inject_wait_timeout): bit 0 arms the decode kernel,
// bit 1 the tcgen05 prefill kernel; off (0) unless a test sets it.
std::atomic<int32_t> g_inject_kernels{0};
std::atomic<uint32_t> g_inject_limit_us{0};

pkv_status fail(pkv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------- device state --

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
uint32_t* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

pkv_status device_state(uint32_t** err_ptr, int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_err_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pkv_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_num_sms[dev] = sms;
        g_err_ptr[dev] = static_cast<uint32_t*>(p);
    }
    if (err_ptr) *err_ptr = g_err_ptr[dev];
    if (num_sms) *num_sms = g_num_sms[dev];
    return PKV_OK;
}

// ------------------------------------------------------------ tensor maps --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    int64_t num_blocks;
    int32_t hkv, d, fp8, dev, kind;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && num_blocks == o.num_blocks && hkv == o.hkv && d == o.d &&
               fp8 == o.fp8 && dev == o.dev && kind == o.kind;
    }
};

// The two tiled views of a pool.
enum MapKind {
    kMapBlockRows = 0,  // {D, 16, Hkv, num_blocks}, box {inner, 16, 1, 1}
    kMapTileRows = 1,   // bf16 only: {64, D/64, 16, Hkv, num_blocks}, box {64, D/64, 16, 1, 1}
    kMapTileGroups = 2, // bf16 only: {64, 8, D/64, 2, num_blocks * Hkv}, box {64, 8, D/64, 2, 1}
};

struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint64_t stamp;
};

constexpr int kMapCache = 16;
thread_local MapEntry g_maps[kMapCache];
thread_local int g_maps_used = 0;
thread_local uint64_t g_map_clock = 0;

// A tiled view of one pool.  kMapBlockRows: dims (innermost first) {D,
// block_size, Hkv, num_blocks}, box {inner, 16, 1, 1}; bf16 rows are split
// into 64-element boxes with the 128-byte swizzle, e4m3 rows are one
// unswizzled box.  kMapTileRows (bf16): one box brings a whole (block, head)
// tile, which costs the TMA unit about two thirds of two half-width boxes.
pkv_status pool_map(const void* pool, const pkv_cache_desc* desc, CUtensorMap* out,
                    MapKind kind = kMapBlockRows) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 0;
    if (fp8) kind = kMapBlockRows;
    const MapKey key{pool, desc->num_blocks, desc->num_kv_heads, desc->head_dim, fp8, dev,
                     static_cast<int32_t>(kind)};
    for (int i = 0; i < g_maps_used; ++i) {
        if (g_maps[i].key == key) {
            g_maps[i].stamp = ++g_map_clock;
            *out = g_maps[i].map;
            return PKV_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const pkv::BoxShape box = pkv::kv_box_shape(desc->head_dim, key.fp8);
    const cuuint64_t elem = key.fp8 ? 1 : 2;
    const cuuint64_t D = static_cast<cuuint64_t>(desc->head_dim);
    const cuuint64_t rows = static_cast<cuuint64_t>(desc->block_size);
    const cuuint64_t hkv = static_cast<cuuint64_t>(desc->num_kv_heads);
    const cuuint64_t nb = static_cast<cuuint64_t>(desc->num_blocks);
    CUtensorMap map;
    CUresult r;
    if (kind == kMapTileGroups) {
        // one box per (block, head) tile, written as [row group g][64-column
        // slice s][8 rows][128 bytes]: every (g, s) slab is one 1024-byte
        // 128-byte-swizzle atom, so the tile is a K-major (K) or MN-major (V)
        // MMA operand whose 8-row groups sit a uniform (D/64) KiB apart, across
        // the tiles of consecutive blocks too
        const cuuint64_t dims[5] = {64, 8, D / 64, 2, nb * hkv};
        const cuuint64_t strides[4] = {D * elem, 64 * elem, 8 * D * elem, rows * D * elem};
        const cuuint32_t boxdim[5] = {64, 8, static_cast<cuuint32_t>(D / 64), 2, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(pool), dims, strides,
               boxdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (kind == kMapTileRows) {
        // one box per (block, head): 16 rows x D/64 slices of 128 bytes, so a
        // row's slices sit side by side (row r, slice h at 128 (r D/64 + h)),
        // each swizzled by its 128-byte unit index
        const cuuint64_t dims[5] = {64, D / 64, rows, hkv, nb};
        const cuuint64_t strides[4] = {64 * elem, D * elem, rows * D * elem, hkv * rows * D * elem};
        const cuuint32_t boxdim[5] = {64, static_cast<cuuint32_t>(D / 64),
                                      static_cast<cuuint32_t>(rows), 1, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(pool), dims, strides,
               boxdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {D, rows, hkv, nb};
        const cuuint64_t strides[3] = {D * elem, D * rows * elem, D * rows * hkv * elem};
        const cuuint32_t boxdim[4] = {static_cast<cuuint32_t>(box.inner),
                                      static_cast<cuuint32_t>(rows), 1, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        r = fn(&map, key.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(pool), dims, strides, boxdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box.swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    int slot = 0;
    if (g_maps_used < kMapCache) {
        slot = g_maps_used++;
    } else {
        for (int i = 1; i < kMapCache; ++i)
            if (g_maps[i].stamp < g_maps[slot].stamp) slot = i;
    }
    g_maps[slot].key = key;
    g_maps[slot].map = map;
    g_maps[slot].stamp = ++g_map_clock;
    *out = map;
    return PKV_OK;
}

// -------------------------------------------------------------- validation --

constexpr int kMaxGroup = 16;
constexpr int kMaxChunk = 256;   // blocks per decode CTA (64 per warp: two ids per lane)
constexpr int kLongChunk = 128;  // the planner's limit unless the batch spans many waves, and
                                 // the e4m3 kernel's (one id per lane)
constexpr int kMinChunk = 32;
constexpr int kMaxSplits = 512;
constexpr int kClusterSplits = 4;  // the decode kernel's cluster-merge limit

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_desc(const pkv_cache_desc* d) {
    if (!d) return fail(PKV_ERR_INVALID_ARG, "desc is NULL");
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0)
        return fail(PKV_ERR_INVALID_ARG, "head counts must be positive (Hq=%d, Hkv=%d)",
                    d->num_q_heads, d->num_kv_heads);
    if (d->num_q_heads % d->num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                    d->num_q_heads, d->num_kv_heads);
    if (d->num_q_heads / d->num_kv_heads > kMaxGroup)
        return fail(PKV_ERR_UNSUPPORTED, "group size %d > %d", d->num_q_heads / d->num_kv_heads,
                    kMaxGroup);
    if (d->head_dim != 64 && d->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", d->head_dim);
    if (d->block_size != 16) return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 16)", d->block_size);
    if (d->kv_dtype != PKV_KV_BF16 && d->kv_dtype != PKV_KV_FP8_E4M3)
        return fail(PKV_ERR_UNSUPPORTED, "kv_dtype %d", d->kv_dtype);
    if (d->num_blocks <= 0 || d->num_blocks > 0x7FFFFFFFLL)
        return fail(PKV_ERR_INVALID_ARG, "num_blocks %lld out of range", (long long)d->num_blocks);
    if (d->max_blocks_per_seq <= 0)
        return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be positive");
    if (d->ring_blocks < 0 || d->ring_blocks > d->max_blocks_per_seq)
        return fail(PKV_ERR_INVALID_ARG, "ring_blocks %d outside [0, max_blocks_per_seq = %d]", d->ring_blocks,
                    d->max_blocks_per_seq);
    if (d->flags & ~(PKV_DESC_PREFETCH_KV | PKV_DESC_INDEPENDENT))
        return fail(PKV_ERR_INVALID_ARG, "unknown desc flags 0x%x", d->flags);
    return PKV_OK;
}

// Decode over a ring cache needs a window whose keys the ring holds: the
// window spans at most ceil((W - 1) / 16) + 1 blocks.  Also the bound on
// max_context_len: the table capacity, or none with a ring.
pkv_status check_ring_window(const pkv_cache_desc* d, int window, int max_context_len) {
    if (d->ring_blocks > 0) {
        if (window <= 0) return fail(PKV_ERR_INVALID_ARG, "a ring cache needs a sliding window");
        if ((window - 1 + d->block_size - 1) / d->block_size + 1 > d->ring_blocks)
            return fail(PKV_ERR_INVALID_ARG, "window %d needs more than ring_blocks = %d blocks", window,
                        d->ring_blocks);
        if (max_context_len < 1) return fail(PKV_ERR_INVALID_ARG, "max_context_len %d < 1", max_context_len);
        return PKV_OK;
    }
    if (max_context_len < 1 || max_context_len > d->max_blocks_per_seq * d->block_size)
        return fail(PKV_ERR_INVALID_ARG, "max_context_len %d outside [1, %d]", max_context_len,
                    d->max_blocks_per_seq * d->block_size);
    return PKV_OK;
}

int elem_bytes(const pkv_cache_desc* d) { return d->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2; }

// ---------------------------------------------------------------- planner --

int max_visible_blocks(int max_ctx, int window) {
    int mb = (max_ctx + 15) / 16;
    if (window > 0) mb = std::min(mb, (window + 14) / 16 + 1);
    return std::max(mb, 1);
}

int resident_ctas(int d, int fp8) {
    // shared memory bound, and the register bound of ~150 registers x 128 threads
    const int smem = pkv::decode_smem_bytes(d, fp8) + 1024;
    return std::max(1, std::min(3, (228 * 1024) / smem));
}

pkv_status plan_decode(const pkv_cache_desc* desc, int num_seqs, int max_ctx, int window,
                       int num_sms, int chunk_req, int* chunk_out, int* splits_out) {
    const int mb = max_visible_blocks(max_ctx, window);
    const int max_chunk = desc->kv_dtype == PKV_KV_FP8_E4M3 ? kLongChunk : kMaxChunk;
    int chunk;
    if (chunk_req > 0) {
        if (chunk_req > max_chunk)
            return fail(PKV_ERR_INVALID_ARG, "chunk_blocks %d > %d", chunk_req, max_chunk);
        chunk = chunk_req;
    } else {
        // Ragged batches average about half their longest context.  Every CTA
        // pays a fixed start (first TMA round trip) and end (combine, partial
        // write, ticket), so aim for one wave of resident CTAs: the fewest,
        // largest chunks that still occupy every slot.
        // Each pair rounds its last chunk up, adding about half a CTA per pair,
        // so size chunks to fill the resident slots without spilling into a
        // second (mostly idle) wave.
        const double pairs = double(num_seqs) * desc->num_kv_heads;
        const double est_blocks = pairs * std::max(1.0, 0.55 * mb);
        const double slots =
            double(std::max(num_sms, 1)) * resident_ctas(desc->head_dim, desc->kv_dtype);
        const double target = std::max(slots - 0.5 * pairs, 0.25 * slots);
        chunk = int(std::ceil(est_blocks / target));
        // Chunks longer than kLongChunk blocks only while the batch still
        // spans at least 8 waves of resident CTAs with them: on the
        // Llama-3-8B-shaped decode (~10 waves at 256 blocks) they measured
        // 0.3 % faster, on the FP8 layer (~3.6 waves at 256 blocks) 23 %
        // slower, its tail of long chunks left alone on the GPU.
        const int cap = pairs * (0.55 * mb / max_chunk + 0.5) >= 8.0 * slots ? max_chunk : kLongChunk;
        chunk = std::max(kMinChunk, std::min(cap, chunk));
        chunk = std::max(chunk, (mb + kMaxSplits - 1) / kMaxSplits);  // bound the split count
        if (chunk > mb) chunk = mb;
        // 2..4 chunks per sequence merge in a thread-block cluster, without
        // the workspace round trip; a plan of 5..8 takes 4 longer chunks
        // instead when they fit one CTA
        const int s = (mb + chunk - 1) / chunk;
        if (s > kClusterSplits && s <= 2 * kClusterSplits && (mb + kClusterSplits - 1) / kClusterSplits <= cap)
            chunk = (mb + kClusterSplits - 1) / kClusterSplits;
    }
    if (chunk > max_chunk)  // more than kMaxSplits chunks of the longest a CTA takes
        return fail(PKV_ERR_UNSUPPORTED, "context of %d blocks needs more than %d chunks of %d blocks", mb,
                    kMaxSplits, max_chunk);
    const int splits = (mb + chunk - 1) / chunk;
    if (splits > kMaxSplits)
        return fail(PKV_ERR_UNSUPPORTED, "context needs %d splits of %d blocks (max %d)", splits, chunk,
                    kMaxSplits);
    *chunk_out = chunk;
    *splits_out = splits;
    return PKV_OK;
}

// The short-query kernel's plan: chunk length in blocks and chunks per
// (sequence, KV head, row tile).  Its CTAs are few next to decode's, so every
// KV range takes the most chunks one cluster merges (kSqMaxSplits): on the
// verify and cascade workloads that measured 1.2-1.3x faster than a one-wave
// plan.  False when the longest KV range does not fit kSqMaxSplits chunks.
bool plan_short_query(int max_kv, int max_q, int window, int* chunk_out, int* splits_out) {
    int mb = std::max(1, (max_kv + 15) / 16);
    if (window > 0) mb = std::min(mb, (window + max_q + 14) / 16 + 1);
    if (mb > pkv::kSqMaxSplits * pkv::kSqMaxChunk) return false;
    const int chunk = (mb + pkv::kSqMaxSplits - 1) / pkv::kSqMaxSplits;
    *chunk_out = chunk;
    *splits_out = (mb + chunk - 1) / chunk;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct DecodeWs {
    size_t counters, lse, o, total;
};

DecodeWs decode_ws_layout(const pkv_cache_desc* d, int num_seqs, int splits) {
    DecodeWs w{};
    const size_t pairs = size_t(num_seqs) * d->num_kv_heads;
    const size_t G = d->num_q_heads / d->num_kv_heads;
    w.counters = 0;
    w.lse = align256(pairs * sizeof(uint32_t));
    w.o = w.lse + align256(pairs * splits * G * sizeof(float));
    w.total = splits > 1 ? w.o + align256(pairs * splits * G * d->head_dim * sizeof(float))
                         : 0;
    return w;
}

}  // namespace

namespace pkv {
BoxShape kv_box_shape(int head_dim, int fp8) {
    if (fp8) return BoxShape{head_dim, 1, 0};
    return BoxShape{64, head_dim / 64, 1};
}
}  // namespace pkv

namespace {

// 3-D tiled view of q [total_q][Hq][D] bf16: box {64, G, QT}, 128-byte swizzle;
// one box is the query tile of one KV group (QT tokens x G heads x 64 columns).
pkv_status q_map(const void* q, int total_q, const pkv_cache_desc* desc, int G, int QT, CUtensorMap* out) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[3] = {cuuint64_t(desc->head_dim), cuuint64_t(desc->num_q_heads), cuuint64_t(total_q)};
    const cuuint64_t strides[2] = {cuuint64_t(desc->head_dim) * 2, cuuint64_t(desc->head_dim) * desc->num_q_heads * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(QT)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (%d)", int(r));
    return PKV_OK;
}

}  // namespace

// ===================================================================== ABI ==

extern "C" {

const char* pkv_last_error(void) { return g_last_error; }

uint64_t pkv_cache_bytes(const pkv_cache_desc* desc) {
    if (check_desc(desc) != PKV_OK) return 0;
    return uint64_t(desc->num_blocks) * desc->num_kv_heads * desc->block_size * desc->head_dim *
           elem_bytes(desc);
}

pkv_status pkv_rope_cos_sin_table(float theta, int32_t rotary_dim, int32_t max_pos,
                                  float* host_out) {
    g_last_error[0] = 0;
    if (!host_out) return fail(PKV_ERR_INVALID_ARG, "host_out is NULL");
    if (rotary_dim <= 0 || rotary_dim % 2 || max_pos < 0 || !(theta > 0.f))
        return fail(PKV_ERR_INVALID_ARG, "bad rope table shape (dim=%d, max_pos=%d, theta=%g)",
                    rotary_dim, max_pos, double(theta));
    const int half = rotary_dim / 2;
    for (int p = 0; p < max_pos; ++p) {
        for (int j = 0; j < half; ++j) {
            const double inv_freq = std::pow(double(theta), -(2.0 * j) / double(rotary_dim));
            const double ang = double(p) * inv_freq;
            host_out[(size_t(p) * half + j) * 2 + 0] = float(std::cos(ang));
            host_out[(size_t(p) * half + j) * 2 + 1] = float(std::sin(ang));
        }
    }
    return PKV_OK;
}

pkv_status pkv_decode_plan(const pkv_cache_desc* desc, int32_t num_seqs, int32_t max_context_len,
                           int32_t window, int32_t num_sms, int32_t* chunk_blocks_out,
                           int32_t* max_splits_out) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (!chunk_blocks_out || !max_splits_out) return fail(PKV_ERR_INVALID_ARG, "null output pointer");
    if (num_seqs < 0 || max_context_len < 1)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d / max_context_len %d", num_seqs, max_context_len);
    if (num_sms <= 0) {
        st = device_state(nullptr, &num_sms);
        if (st != PKV_OK) return st;
    }
    int c = 0, s = 0;
    st = plan_decode(desc, num_seqs, max_context_len, window, num_sms, 0, &c, &s);
    if (st != PKV_OK) return st;
    *chunk_blocks_out = c;
    *max_splits_out = s;
    return PKV_OK;
}

size_t pkv_decode_workspace_size(const pkv_cache_desc* desc, int32_t num_seqs,
                                 int32_t max_context_len, int32_t window, int32_t chunk_blocks) {
    if (check_desc(desc) != PKV_OK || num_seqs <= 0 || max_context_len < 1) return 0;
    int sms = 0;
    if (chunk_blocks <= 0 && device_state(nullptr, &sms) != PKV_OK) return 0;
    int c = 0, s = 0;
    if (plan_decode(desc, num_seqs, max_context_len, window, sms, chunk_blocks, &c, &s) != PKV_OK)
        return 0;
    return decode_ws_layout(desc, num_seqs, s).total;
}

}  // extern "C"

namespace {

// The new token of a decode step (pkv_decode_step); null for plain decode.
struct StepIn {
    const void* k_new;
    const void* v_new;
    const float* cos_sin;
    int32_t max_pos;
};

// Where the decode's split states live: the caller's workspace, or the
// library's fixed scratch array (pkv_decode_attention_static).
enum class Scratch { kCaller, kStatic };

pkv_status static_scratch(void** out, size_t* bytes);

pkv_status decode_impl(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                       const void* v_cache, const float* k_scale, const float* v_scale,
                       const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                       int32_t max_context_len, float sm_scale, int32_t window, const float* sinks,
                       int32_t chunk_blocks, void* out, float* lse_out, void* workspace,
                       size_t workspace_bytes, pkv_stream_t stream, const StepIn* step,
                       Scratch scratch = Scratch::kCaller) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || num_seqs > 65535)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d out of range [0, 65535]", num_seqs);
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    const bool fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3;
    if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    st = check_ring_window(desc, window, max_context_len);
    if (st != PKV_OK) return st;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the pools must be 16-byte aligned");
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
    if (step) {
        if (!step->k_new || !step->v_new) return fail(PKV_ERR_INVALID_ARG, "k_new / v_new is NULL");
        if (!aligned(step->k_new, 16) || !aligned(step->v_new, 16))
            return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
        if (step->cos_sin) {
            if (!aligned(step->cos_sin, 16)) return fail(PKV_ERR_INVALID_ARG, "rope_cos_sin must be 16-byte aligned");
            // the new token sits at context_lens[s] - 1 <= max_context_len - 1
            if (step->max_pos < max_context_len)
                return fail(PKV_ERR_INVALID_ARG, "rope_max_pos %d < max_context_len %d", step->max_pos,
                            max_context_len);
        }
    }
    uint32_t* err = nullptr;
    int sms = 0;
    st = device_state(&err, &sms);
    if (st != PKV_OK) return st;
    int chunk = 0, splits = 0;
    st = plan_decode(desc, num_seqs, max_context_len, window, sms, chunk_blocks, &chunk, &splits);
    if (st != PKV_OK) return st;
    const DecodeWs ws = decode_ws_layout(desc, num_seqs, splits);
    if (scratch == Scratch::kStatic) {
        size_t cap = 0;
        st = static_scratch(&workspace, &cap);
        if (st != PKV_OK) return st;
        if (ws.total > cap)
            return fail(PKV_ERR_WORKSPACE,
                        "this batch needs %zu bytes of decode scratch, more than the %zu-byte static "
                        "array; use pkv_decode_attention with a workspace, or a larger chunk_blocks",
                        ws.total, cap);
        workspace_bytes = cap;
    }
    if (ws.total > 0) {
        if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", ws.total);
        if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        if (workspace_bytes < ws.total)
            return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, ws.total);
    }
    CUtensorMap kmap, vmap;
    st = pool_map(k_cache, desc, &kmap, kMapTileRows);
    if (st != PKV_OK) return st;
    st = pool_map(v_cache, desc, &vmap, kMapTileRows);
    if (st != PKV_OK) return st;
    if (scratch == Scratch::kStatic && ws.total > 0 && pkv::decode_uses_tickets(splits)) {
        // The static array keeps whatever the last call left there, which may
        // be another layout's partial states: a plan that merges through
        // tickets clears them first (cluster plans never read them).
        const size_t pairs = size_t(num_seqs) * desc->num_kv_heads;
        cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(workspace) + ws.counters, 0,
                                        pairs * sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "clear static decode tickets");
    }
    pkv::DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.sinks = sinks;
    a.ring = desc->ring_blocks;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    a.counters = ws.total ? reinterpret_cast<uint32_t*>(wsb + ws.counters) : nullptr;
    a.part_lse = ws.total ? reinterpret_cast<float*>(wsb + ws.lse) : nullptr;
    a.part_o = ws.total ? reinterpret_cast<float*>(wsb + ws.o) : nullptr;
    a.err = err;
    a.num_seqs = num_seqs;
    a.hq = desc->num_q_heads;
    a.hkv = desc->num_kv_heads;
    a.group = desc->num_q_heads / desc->num_kv_heads;
    a.d = desc->head_dim;
    a.mbps = desc->max_blocks_per_seq;
    a.window = window;
    a.chunk_blocks = chunk;
    a.max_splits = splits;
    a.max_ctx = max_context_len;
    a.fp8 = fp8 ? 1 : 0;
    a.num_blocks = desc->num_blocks;
    a.sm_scale = sm_scale;
    a.inject_timeout = g_inject_kernels.load() & 1;
    a.inject_limit_us = g_inject_limit_us.load();
    a.early_kv = (desc->flags & PKV_DESC_PREFETCH_KV) ? 1 : 0;
    a.defer_wait = (desc->flags & PKV_DESC_INDEPENDENT) ? 1 : 0;
    if (step) {
        a.k_new = step->k_new;
        a.v_new = step->v_new;
        a.cos_sin = step->cos_sin;
        a.k_pool = const_cast<void*>(k_cache);
        a.v_pool = const_cast<void*>(v_cache);
    }
    cudaError_t e = pkv::launch_decode(a, kmap, vmap, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, step ? "decode step launch" : "decode launch");
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                                const void* v_cache, const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int32_t num_seqs, int32_t max_context_len, float sm_scale,
                                int32_t window, const float* sinks, int32_t chunk_blocks, void* out,
                                float* lse_out, void* workspace, size_t workspace_bytes,
                                pkv_stream_t stream) {
    return decode_impl(desc, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                       max_context_len, sm_scale, window, sinks, chunk_blocks, out, lse_out, workspace,
                       workspace_bytes, stream, nullptr);
}

pkv_status pkv_decode_step(const pkv_cache_desc* desc, const void* q, const void* k_new,
                           const void* v_new, const float* rope_cos_sin, int32_t rope_max_pos,
                           void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
                           int32_t max_context_len, float sm_scale, int32_t window, const float* sinks,
                           int32_t chunk_blocks, void* out, float* lse_out, void* workspace,
                           size_t workspace_bytes, pkv_stream_t stream) {
    const StepIn step{k_new, v_new, rope_cos_sin, rope_max_pos};
    return decode_impl(desc, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                       max_context_len, sm_scale, window, sinks, chunk_blocks, out, lse_out, workspace,
                       workspace_bytes, stream, &step);
}

size_t pkv_prefill_workspace_size(const pkv_cache_desc* desc, int32_t num_seqs,
                                  int32_t total_q_tokens) {
    // every prefill path reads the pools (bf16 or e4m3) directly
    (void)desc;
    (void)num_seqs;
    (void)total_q_tokens;
    return 0;
}

}  // extern "C"

namespace {

// The ragged prefill.  scaled_codes: the bf16 pools hold e4m3 codes widened
// exactly (a staged e4m3 cache); k_scale / v_scale are then folded in as for
// an e4m3 pool.
pkv_status prefill_impl(const pkv_cache_desc* desc, const void* q, const int32_t* qo_indptr,
                        const void* k_cache, const void* v_cache, const float* k_scale,
                        const float* v_scale, const int32_t* block_tables, const int32_t* kv_lens,
                        int32_t num_seqs, int32_t total_q_tokens, const int32_t* qo_indptr_host,
                        const int32_t* kv_lens_host, float sm_scale, int32_t causal, int32_t window,
                        void* out, float* lse_out, pkv_stream_t stream, bool scaled_codes) {
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (desc->ring_blocks > 0)
        return fail(PKV_ERR_UNSUPPORTED, "prefill reads linear tables; a ring cache takes pkv_prefill_ring_commit");
    const bool fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3;
    if (scaled_codes && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "scaled codes need k_scale and v_scale");
    if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    if (num_seqs < 0 || num_seqs > 65535)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d out of range [0, 65535]", num_seqs);
    if (total_q_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "total_q_tokens < 0");
    if (num_seqs == 0 || total_q_tokens == 0) return PKV_OK;
    if (!q || !qo_indptr || !k_cache || !v_cache || !block_tables || !kv_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the pools must be 16-byte aligned");
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
    const int G = desc->num_q_heads / desc->num_kv_heads;
    const int QT = pkv::prefill_tc_q_tile(G);
    int max_q = total_q_tokens;
    if (qo_indptr_host) {
        if (qo_indptr_host[0] != 0 || qo_indptr_host[num_seqs] != total_q_tokens)
            return fail(PKV_ERR_INVALID_ARG, "qo_indptr_host must run from 0 to total_q_tokens");
        max_q = 0;
        for (int s = 0; s < num_seqs; ++s) {
            const int ql = qo_indptr_host[s + 1] - qo_indptr_host[s];
            if (ql < 0) return fail(PKV_ERR_INVALID_ARG, "qo_indptr_host decreases at %d", s);
            max_q = std::max(max_q, ql);
            if (kv_lens_host) {
                if (kv_lens_host[s] < ql)
                    return fail(PKV_ERR_INVALID_ARG, "sequence %d: kv_len %d < q_len %d", s, kv_lens_host[s], ql);
                if (kv_lens_host[s] > desc->max_blocks_per_seq * desc->block_size)
                    return fail(PKV_ERR_INVALID_ARG, "sequence %d: kv_len %d beyond the table", s, kv_lens_host[s]);
            }
        }
    }
    const int max_qtiles = (max_q + QT - 1) / QT;
    if (max_qtiles == 0) return PKV_OK;
    uint32_t* err = nullptr;
    st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    // at most 64 query rows (tokens x heads of a group) per sequence: the
    // decode-shaped short-query kernel (needs the host query lengths)
    int sq_chunk = 0, sq_splits = 0;
    int kv_bound = desc->max_blocks_per_seq * desc->block_size;
    if (kv_lens_host) {
        kv_bound = 0;
        for (int s2 = 0; s2 < num_seqs; ++s2) kv_bound = std::max(kv_bound, kv_lens_host[s2]);
    }
    const bool short_q = qo_indptr_host && max_q * G <= pkv::kSqMaxRowTiles * 16 &&
                         plan_short_query(kv_bound, max_q, window, &sq_chunk, &sq_splits);
    // e4m3 pools: both kernels read the codes and convert them on chip (the
    // tcgen05 kernel into f16 tiles in shared memory, the short-query kernel
    // into f16 MMA fragments), with the scales folded in; no workspace
    pkv::PrefillArgs a{};
    a.k_scale = fp8 || scaled_codes ? k_scale : nullptr;
    a.v_scale = fp8 || scaled_codes ? v_scale : nullptr;
    a.q = q;
    a.out = out;
    a.lse_out = lse_out;
    a.qo_indptr = qo_indptr;
    a.kv_lens = kv_lens;
    a.block_tables = block_tables;
    a.err = err;
    a.num_seqs = num_seqs;
    a.hq = desc->num_q_heads;
    a.hkv = desc->num_kv_heads;
    a.group = G;
    a.d = desc->head_dim;
    a.mbps = desc->max_blocks_per_seq;
    a.causal = causal ? 1 : 0;
    a.window = window;
    a.max_qtiles = max_qtiles;
    a.q_tile = QT;
    a.total_q = total_q_tokens;
    a.num_blocks = desc->num_blocks;
    a.sm_scale = sm_scale;
    if (qo_indptr_host && kv_lens_host && num_seqs <= pkv::kPrefillOrderMax) {
        // dispatch the sequences with the most causal work first: key-query
        // pairs q (kv - q) + q (q + 1) / 2 of each sequence
        std::vector<std::pair<int64_t, int>> work(static_cast<size_t>(num_seqs));
        for (int s = 0; s < num_seqs; ++s) {
            const int64_t ql = qo_indptr_host[s + 1] - qo_indptr_host[s];
            const int64_t kl = kv_lens_host[s];
            work[static_cast<size_t>(s)] = {-(ql * (kl - ql) + ql * (ql + 1) / 2), s};
        }
        std::stable_sort(work.begin(), work.end());
        for (int i = 0; i < num_seqs; ++i) a.seq_order[i] = static_cast<uint16_t>(work[static_cast<size_t>(i)].second);
        a.ordered = 1;
    }
    if (short_q) {
        CUtensorMap tkmap, tvmap;
        st = pool_map(k_cache, desc, &tkmap, kMapTileRows);
        if (st != PKV_OK) return st;
        st = pool_map(v_cache, desc, &tvmap, kMapTileRows);
        if (st != PKV_OK) return st;
        a.sq_chunk = sq_chunk;
        a.sq_splits = sq_splits;
        a.sq_row_tiles = (max_q * G + 15) / 16;
        a.fp8 = fp8 ? 1 : 0;
        cudaError_t e = pkv::launch_short_query(a, tkmap, tvmap, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "short-query launch");
        return PKV_OK;
    }
    // tcgen05 kernel: bf16 pools through the tile-group view (one 128-byte
    // swizzled box per (block, head), already an MMA operand); e4m3 pools
    // through the row view (one unswizzled box of codes per (block, head))
    CUtensorMap kmap, vmap, qmap;
    st = pool_map(k_cache, desc, &kmap, fp8 ? kMapBlockRows : kMapTileGroups);
    if (st != PKV_OK) return st;
    st = pool_map(v_cache, desc, &vmap, fp8 ? kMapBlockRows : kMapTileGroups);
    if (st != PKV_OK) return st;
    st = q_map(q, total_q_tokens, desc, G, QT, &qmap);
    if (st != PKV_OK) return st;
    a.fp8 = fp8 ? 1 : 0;
    a.inject_timeout = (g_inject_kernels.load() >> 1) & 1;
    a.inject_limit_us = g_inject_limit_us.load();
    cudaError_t e = pkv::launch_prefill_tc(a, qmap, kmap, vmap, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PKV_OK;
}

// Staging blocks per sequence of a ring-cache prefill: the chunk's window
// reaches window - 1 keys before its first token, from a block boundary.
int ring_stage_cap(int window, int max_q) { return (window - 1 + max_q + 15) / 16 + 1; }

struct RingWs {
    size_t tables, lens, k, v, total;
};
RingWs ring_ws_layout(const pkv_cache_desc* d, int num_seqs, int cap) {
    RingWs w{};
    const size_t blocks = size_t(num_seqs) * cap;
    const size_t block_bytes = size_t(d->num_kv_heads) * d->block_size * d->head_dim * 2;
    w.tables = 0;
    w.lens = align256(blocks * sizeof(int32_t));
    w.k = w.lens + align256(size_t(num_seqs) * sizeof(int32_t));
    w.v = w.k + align256(blocks * block_bytes);
    w.total = w.v + align256(blocks * block_bytes);
    return w;
}

}  // namespace

extern "C" {

pkv_status pkv_prefill_attention_ragged(const pkv_cache_desc* desc, const void* q,
                                        const int32_t* qo_indptr, const void* k_cache,
                                        const void* v_cache, const float* k_scale,
                                        const float* v_scale, const int32_t* block_tables,
                                        const int32_t* kv_lens, int32_t num_seqs,
                                        int32_t total_q_tokens, const int32_t* qo_indptr_host,
                                        const int32_t* kv_lens_host, float sm_scale,
                                        int32_t causal, int32_t window, void* out,
                                        float* lse_out, void* workspace,
                                        size_t workspace_bytes, pkv_stream_t stream) {
    g_last_error[0] = 0;
    (void)workspace;  // no prefill path needs one (pkv_prefill_workspace_size is 0)
    (void)workspace_bytes;
    return prefill_impl(desc, q, qo_indptr, k_cache, v_cache, k_scale, v_scale, block_tables, kv_lens,
                        num_seqs, total_q_tokens, qo_indptr_host, kv_lens_host, sm_scale, causal, window,
                        out, lse_out, stream, false);
}

size_t pkv_prefill_ring_workspace_size(const pkv_cache_desc* desc, int32_t num_seqs, int32_t window,
                                       int32_t max_q_len) {
    if (check_desc(desc) != PKV_OK || num_seqs <= 0 || window <= 0 || max_q_len < 1) return 0;
    return ring_ws_layout(desc, num_seqs, ring_stage_cap(window, max_q_len)).total;
}

pkv_status pkv_prefill_ring_commit(const pkv_cache_desc* desc, const void* q, const int32_t* qo_indptr,
                                   const void* k_chunk, const void* v_chunk, void* k_cache, void* v_cache,
                                   const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                   const int32_t* kv_lens, int32_t num_seqs, int32_t total_q_tokens,
                                   const int32_t* qo_indptr_host, const int32_t* kv_lens_host,
                                   float sm_scale, int32_t window, void* out, float* lse_out,
                                   void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (desc->ring_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "pkv_prefill_ring_commit needs a ring cache");
    const bool fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3;
    if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    if (num_seqs < 0 || num_seqs > 65535)
        return fail(PKV_ERR_INVALID_ARG, "num_seqs %d out of range [0, 65535]", num_seqs);
    if (total_q_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "total_q_tokens < 0");
    if (num_seqs == 0 || total_q_tokens == 0) return PKV_OK;
    if (!q || !qo_indptr || !k_chunk || !v_chunk || !k_cache || !v_cache || !block_tables || !kv_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    if (!qo_indptr_host || !kv_lens_host)
        return fail(PKV_ERR_INVALID_ARG, "a ring-cache prefill needs qo_indptr_host and kv_lens_host");
    // a window the ring holds: any position's window fits in ring_blocks blocks
    st = check_ring_window(desc, window, 1);
    if (st != PKV_OK) return st;
    if (qo_indptr_host[0] != 0 || qo_indptr_host[num_seqs] != total_q_tokens)
        return fail(PKV_ERR_INVALID_ARG, "qo_indptr_host must run from 0 to total_q_tokens");
    int max_q = 0;
    std::vector<int32_t> stage_lens_host(static_cast<size_t>(num_seqs));
    for (int s = 0; s < num_seqs; ++s) {
        const int ql = qo_indptr_host[s + 1] - qo_indptr_host[s];
        if (ql < 0) return fail(PKV_ERR_INVALID_ARG, "qo_indptr_host decreases at %d", s);
        if (kv_lens_host[s] < ql) return fail(PKV_ERR_INVALID_ARG, "sequence %d: kv_len %d < q_len %d", s,
                                              kv_lens_host[s], ql);
        max_q = std::max(max_q, ql);
        const int lo = std::max(0, kv_lens_host[s] - ql - window + 1);
        stage_lens_host[static_cast<size_t>(s)] = kv_lens_host[s] - (lo - lo % 16);
    }
    const int cap = ring_stage_cap(window, max_q);
    const RingWs ws = ring_ws_layout(desc, num_seqs, cap);
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", ws.total);
    if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < ws.total)
        return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, ws.total);
    if (int64_t(num_seqs) * cap > 0x7FFFFFFFLL) return fail(PKV_ERR_UNSUPPORTED, "staging table too large");
    uint32_t* err = nullptr;
    st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    pkv::RingStageArgs g{};
    g.k_cache = k_cache;
    g.v_cache = v_cache;
    g.k_scale = k_scale;
    g.v_scale = v_scale;
    g.block_tables = block_tables;
    g.qo_indptr = qo_indptr;
    g.kv_lens = kv_lens;
    g.k_chunk = k_chunk;
    g.v_chunk = v_chunk;
    g.stage_tables = reinterpret_cast<int32_t*>(wsb + ws.tables);
    g.stage_lens = reinterpret_cast<int32_t*>(wsb + ws.lens);
    g.k_stage = reinterpret_cast<uint16_t*>(wsb + ws.k);
    g.v_stage = reinterpret_cast<uint16_t*>(wsb + ws.v);
    g.k_ring_out = k_cache;
    g.v_ring_out = v_cache;
    g.num_seqs = num_seqs;
    g.hkv = desc->num_kv_heads;
    g.d = desc->head_dim;
    g.mbps = desc->max_blocks_per_seq;
    g.ring = desc->ring_blocks;
    g.window = window;
    g.cap = cap;
    g.fp8 = fp8 ? 1 : 0;
    g.total_q = total_q_tokens;
    g.num_blocks = desc->num_blocks;
    g.err = err;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // 1. the window's keys, ring and chunk, into a linear bf16 staging copy
    cudaError_t e = pkv::launch_stage_ring(g, s);
    if (e != cudaSuccess) return cuda_fail(e, "ring staging launch");
    // 2. the stream-ordered cache commit: the chunk's surviving tokens into the ring
    e = pkv::launch_commit_ring(g, s);
    if (e != cudaSuccess) return cuda_fail(e, "ring commit launch");
    // 3. the ragged prefill over the staging copy
    pkv_cache_desc staged = *desc;
    staged.kv_dtype = PKV_KV_BF16;
    staged.ring_blocks = 0;
    staged.num_blocks = static_cast<int64_t>(num_seqs) * cap;
    staged.max_blocks_per_seq = cap;
    return prefill_impl(&staged, q, qo_indptr, g.k_stage, g.v_stage, k_scale, v_scale, g.stage_tables,
                        g.stage_lens, num_seqs, total_q_tokens, qo_indptr_host, stage_lens_host.data(),
                        sm_scale, 1, window, out, lse_out, stream, fp8);
}

pkv_status pkv_append_rope(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                           const float* k_scale, const float* v_scale,
                           const int32_t* block_tables, int32_t num_seqs,
                           const int32_t* token_to_seq, const int32_t* positions,
                           int32_t num_tokens, const void* k_new, const void* v_new,
                           void* q_inout, const float* rope_cos_sin, int32_t rope_max_pos,
                           pkv_stream_t stream) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_tokens < 0 || num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "negative count");
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !block_tables || !token_to_seq || !positions || !k_new || !v_new)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    const bool fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3;
    if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    if (rope_cos_sin && rope_max_pos <= 0) return fail(PKV_ERR_INVALID_ARG, "rope_max_pos must be positive");
    uint32_t* err = nullptr;
    st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    pkv::AppendArgs a{};
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.token_to_seq = token_to_seq;
    a.positions = positions;
    a.k_new = k_new;
    a.v_new = v_new;
    a.q = q_inout;
    a.cos_sin = rope_cos_sin;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.hq = desc->num_q_heads;
    a.hkv = desc->num_kv_heads;
    a.d = desc->head_dim;
    a.mbps = desc->max_blocks_per_seq;
    a.max_pos = rope_max_pos;
    a.ring = desc->ring_blocks;
    a.num_blocks = desc->num_blocks;
    a.fp8 = fp8 ? 1 : 0;
    a.err = err;
    cudaError_t e = pkv::launch_append_rope(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return PKV_OK;
}

pkv_status pkv_gather_kv(const pkv_cache_desc* desc, const void* cache, const int32_t* block_tables,
                         const int32_t* context_lens, const int32_t* cu_context_lens,
                         int32_t num_seqs, int64_t total_tokens, void* out, pkv_stream_t stream) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (desc->ring_blocks > 0) return fail(PKV_ERR_UNSUPPORTED, "gather reads linear tables (no ring cache)");
    if (num_seqs < 0 || total_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "negative count");
    if (num_seqs == 0 || total_tokens == 0) return PKV_OK;
    if (!cache || !block_tables || !context_lens || !cu_context_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    if (!aligned(cache, 16) || !aligned(out, 16))
        return fail(PKV_ERR_INVALID_ARG, "cache and out must be 16-byte aligned");
    uint32_t* err = nullptr;
    st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    pkv::GatherArgs a{};
    a.cache = cache;
    a.block_tables = block_tables;
    a.lens = context_lens;
    a.cu_lens = cu_context_lens;
    a.out = out;
    a.num_seqs = num_seqs;
    a.hkv = desc->num_kv_heads;
    a.row_bytes = desc->head_dim * elem_bytes(desc);
    a.mbps = desc->max_blocks_per_seq;
    a.total_tokens = total_tokens;
    a.num_blocks = desc->num_blocks;
    a.err = err;
    cudaError_t e = pkv::launch_gather(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    return PKV_OK;
}

pkv_status pkv_copy_blocks(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                           const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                           pkv_stream_t stream) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (num_pairs < 0 || num_pairs > 0x7FFFFFFF / 2) return fail(PKV_ERR_INVALID_ARG, "num_pairs %d", num_pairs);
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_blocks || !dst_blocks)
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(PKV_ERR_INVALID_ARG, "the pools must be 16-byte aligned");
    uint32_t* err = nullptr;
    st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    pkv::CopyArgs a{};
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.src = src_blocks;
    a.dst = dst_blocks;
    a.num_pairs = num_pairs;
    a.num_blocks = desc->num_blocks;
    a.block_bytes = int64_t(desc->num_kv_heads) * desc->block_size * desc->head_dim * elem_bytes(desc);
    a.err = err;
    cudaError_t e = pkv::launch_copy_blocks(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "copy launch");
    return PKV_OK;
}

pkv_status pkv_merge_states(const float* o_parts, const float* lse_parts, int32_t num_parts,
                            int32_t num_rows, int32_t num_heads, int32_t head_dim, void* out,
                            float* lse_out, pkv_stream_t stream) {
    g_last_error[0] = 0;
    if (num_parts < 0 || num_rows < 0 || num_heads < 0 || head_dim <= 0)
        return fail(PKV_ERR_INVALID_ARG, "bad merge shape");
    if (num_rows == 0 || num_heads == 0) return PKV_OK;
    if (!out || (num_parts > 0 && (!o_parts || !lse_parts)))
        return fail(PKV_ERR_INVALID_ARG, "null device pointer");
    pkv::MergeArgs a{o_parts, lse_parts, out, lse_out, num_parts, num_rows, num_heads, head_dim};
    cudaError_t e = pkv::launch_merge(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return PKV_OK;
}

// ---------------------------------------------------- cascade decode (f2) --
//
// The queries of a group of consecutive sequences that share a cached prefix
// attend that prefix in one pass of the prefill kernel (not causal: every
// query sees the whole prefix), which reads each prefix block once for the
// whole group; each sequence's own suffix goes through the decode kernel;
// the two fp32 (o, lse) states merge exactly as split-KV partials do.
// e4m3 pools: the prefix pass reads the codes and folds the scales in, as
// the prefill does.  With a sliding window a query
// sees at most window - 1 prefix keys, the last ones before its suffix, and
// they differ per sequence: the prefix pass is then the decode kernel over
// the group's prefix table with each sequence's own window start.

namespace {
struct CascadeWs {
    size_t o, lse, dec, dec_bytes, pre, pre_bytes, total;
};
CascadeWs cascade_ws_layout(const pkv_cache_desc* d, int num_groups, int num_seqs, int max_prefix_len,
                            int max_suffix_len, int window, int sms) {
    CascadeWs w{};
    const size_t rows = size_t(num_seqs) * d->num_q_heads;
    w.o = 0;
    w.lse = align256(2 * rows * d->head_dim * sizeof(float));
    w.dec = w.lse + align256(2 * rows * sizeof(float));
    int c = 0, sp = 0;
    if (plan_decode(d, num_seqs, std::max(max_suffix_len, 1), window, sms, 0, &c, &sp) == PKV_OK)
        w.dec_bytes = decode_ws_layout(d, num_seqs, sp).total;
    w.pre = w.dec + align256(w.dec_bytes);
    if (window > 0 && max_prefix_len > 0 &&
        plan_decode(d, num_seqs, max_prefix_len, window, sms, 0, &c, &sp) == PKV_OK)
        w.pre_bytes = decode_ws_layout(d, num_seqs, sp).total;
    w.total = w.pre + align256(w.pre_bytes);
    (void)num_groups;
    return w;
}
}  // namespace

size_t pkv_cascade_workspace_size(const pkv_cache_desc* desc, int32_t num_groups, int32_t num_seqs,
                                  int32_t max_prefix_len, int32_t max_suffix_len, int32_t window) {
    if (check_desc(desc) != PKV_OK || num_groups <= 0 || num_seqs <= 0 || max_suffix_len < 1 ||
        max_prefix_len < 0)
        return 0;
    int sms = 0;
    if (device_state(nullptr, &sms) != PKV_OK) return 0;
    return cascade_ws_layout(desc, num_groups, num_seqs, max_prefix_len, max_suffix_len, window, sms).total;
}

pkv_status pkv_cascade_decode(const pkv_cache_desc* desc, const void* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              int32_t num_groups, const int32_t* group_indptr,
                              const int32_t* group_indptr_host, const int32_t* prefix_tables,
                              const int32_t* prefix_lens, const int32_t* prefix_lens_host,
                              int32_t num_seqs, const int32_t* suffix_tables,
                              const int32_t* suffix_lens, int32_t max_suffix_len, float sm_scale,
                              int32_t window, void* out, float* lse_out, void* workspace,
                              size_t workspace_bytes, pkv_stream_t stream) {
    g_last_error[0] = 0;
    pkv_status st = check_desc(desc);
    if (st != PKV_OK) return st;
    if (desc->ring_blocks > 0) return fail(PKV_ERR_UNSUPPORTED, "cascade decode reads linear tables (no ring cache)");
    const bool fp8 = desc->kv_dtype == PKV_KV_FP8_E4M3;
    if (fp8 && (!k_scale || !v_scale)) return fail(PKV_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    if (num_seqs < 0 || num_seqs > 65535) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d out of range", num_seqs);
    if (num_seqs == 0) return PKV_OK;
    if (num_groups < 1 || num_groups > num_seqs)
        return fail(PKV_ERR_INVALID_ARG, "num_groups %d outside [1, num_seqs]", num_groups);
    if (!q || !k_cache || !v_cache || !group_indptr || !group_indptr_host || !prefix_tables || !prefix_lens ||
        !prefix_lens_host || !suffix_tables || !suffix_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(PKV_ERR_INVALID_ARG, "q, out and the pools must be 16-byte aligned");
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
    const int cap = desc->max_blocks_per_seq * desc->block_size;
    if (max_suffix_len < 1 || max_suffix_len > cap)
        return fail(PKV_ERR_INVALID_ARG, "max_suffix_len %d outside [1, %d]", max_suffix_len, cap);
    if (group_indptr_host[0] != 0 || group_indptr_host[num_groups] != num_seqs)
        return fail(PKV_ERR_INVALID_ARG, "group_indptr_host must run from 0 to num_seqs");
    int max_group = 0, max_prefix = 0;
    for (int g = 0; g < num_groups; ++g) {
        const int n = group_indptr_host[g + 1] - group_indptr_host[g];
        if (n < 0) return fail(PKV_ERR_INVALID_ARG, "group_indptr_host decreases at %d", g);
        max_group = std::max(max_group, n);
        if (prefix_lens_host[g] < 0 || prefix_lens_host[g] > cap)
            return fail(PKV_ERR_INVALID_ARG, "group %d: prefix length %d outside [0, %d]", g, prefix_lens_host[g], cap);
        max_prefix = std::max(max_prefix, prefix_lens_host[g]);
    }
    uint32_t* err = nullptr;
    int sms = 0;
    st = device_state(&err, &sms);
    if (st != PKV_OK) return st;
    const CascadeWs ws = cascade_ws_layout(desc, num_groups, num_seqs, max_prefix, max_suffix_len, window, sms);
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", ws.total);
    if (!aligned(workspace, 256)) return fail(PKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (workspace_bytes < ws.total)
        return fail(PKV_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, ws.total);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    float* o_parts = reinterpret_cast<float*>(wsb + ws.o);    // [2][num_seqs][Hq][D]
    float* lse_parts = reinterpret_cast<float*>(wsb + ws.lse);  // [2][num_seqs][Hq]
    const size_t rows = size_t(num_seqs) * desc->num_q_heads;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int G = desc->num_q_heads / desc->num_kv_heads;

    // part 0: every group's queries over its shared prefix
    bool prefix_launched = false;
    if (window > 0 && max_prefix > 0) {
        // each sequence over the prefix keys its window reaches (decode kernel)
        int chunk = 0, splits = 0;
        st = plan_decode(desc, num_seqs, max_prefix, window, sms, 0, &chunk, &splits);
        if (st != PKV_OK) return st;
        const DecodeWs dws = decode_ws_layout(desc, num_seqs, splits);
        CUtensorMap kmap, vmap;
        st = pool_map(k_cache, desc, &kmap, kMapTileRows);
        if (st != PKV_OK) return st;
        st = pool_map(v_cache, desc, &vmap, kMapTileRows);
        if (st != PKV_OK) return st;
        uint8_t* dwb = wsb + ws.pre;
        pkv::DecodeArgs a{};
        a.q = q;
        a.out_f32 = o_parts;
        a.lse_out = lse_parts;
        a.block_tables = prefix_tables;
        a.context_lens = prefix_lens;
        a.group_indptr = group_indptr;
        a.group_suffix_lens = suffix_lens;
        a.num_groups = num_groups;
        a.k_scale = k_scale;
        a.v_scale = v_scale;
        a.counters = dws.total ? reinterpret_cast<uint32_t*>(dwb + dws.counters) : nullptr;
        a.part_lse = dws.total ? reinterpret_cast<float*>(dwb + dws.lse) : nullptr;
        a.part_o = dws.total ? reinterpret_cast<float*>(dwb + dws.o) : nullptr;
        a.err = err;
        a.num_seqs = num_seqs;
        a.hq = desc->num_q_heads;
        a.hkv = desc->num_kv_heads;
        a.group = G;
        a.d = desc->head_dim;
        a.mbps = desc->max_blocks_per_seq;
        a.window = window;
        a.chunk_blocks = chunk;
        a.max_splits = splits;
        a.max_ctx = max_prefix;
        a.fp8 = fp8 ? 1 : 0;
        a.num_blocks = desc->num_blocks;
        a.sm_scale = sm_scale;
        cudaError_t e = pkv::launch_decode(a, kmap, vmap, s);
        if (e != cudaSuccess) return cuda_fail(e, "cascade prefix launch");
        prefix_launched = true;
    } else if (window <= 0) {
        const int QT = pkv::prefill_tc_q_tile(G);
        // a group's queries (at most 64 rows) over its prefix: the short-query
        // kernel; more: the tcgen05 prefill (non-causal, fp32 state out)
        const int max_qtiles = (max_group + QT - 1) / QT;
        int sq_chunk = 0, sq_splits = 0;
        const bool short_q = max_qtiles > 0 && max_group * G <= pkv::kSqMaxRowTiles * 16 &&
                             plan_short_query(max_prefix, max_group, -1, &sq_chunk, &sq_splits);
        // e4m3 pools: either kernel converts the codes on chip, scales folded in
        pkv::PrefillArgs a{};
        a.q = q;
        a.k_scale = fp8 ? k_scale : nullptr;
        a.v_scale = fp8 ? v_scale : nullptr;
        a.out = nullptr;
        a.out_f32 = o_parts;
        a.lse_out = lse_parts;
        a.qo_indptr = group_indptr;
        a.kv_lens = prefix_lens;
        a.block_tables = prefix_tables;
        a.err = err;
        a.num_seqs = num_groups;
        a.hq = desc->num_q_heads;
        a.hkv = desc->num_kv_heads;
        a.group = G;
        a.d = desc->head_dim;
        a.mbps = desc->max_blocks_per_seq;
        a.causal = 0;
        a.window = -1;
        a.max_qtiles = max_qtiles;
        a.q_tile = QT;
        a.total_q = num_seqs;
        a.num_blocks = desc->num_blocks;
        a.sm_scale = sm_scale;
        if (short_q) {
            CUtensorMap tkmap, tvmap;
            st = pool_map(k_cache, desc, &tkmap, kMapTileRows);
            if (st != PKV_OK) return st;
            st = pool_map(v_cache, desc, &tvmap, kMapTileRows);
            if (st != PKV_OK) return st;
            a.sq_chunk = sq_chunk;
            a.sq_splits = sq_splits;
            a.sq_row_tiles = (max_group * G + 15) / 16;
            a.fp8 = fp8 ? 1 : 0;
            cudaError_t e = pkv::launch_short_query(a, tkmap, tvmap, s);
            if (e != cudaSuccess) return cuda_fail(e, "cascade prefix launch");
            prefix_launched = true;
        } else if (max_qtiles > 0) {
            CUtensorMap kmap, vmap, qmap;
            st = pool_map(k_cache, desc, &kmap, fp8 ? kMapBlockRows : kMapTileGroups);
            if (st != PKV_OK) return st;
            st = pool_map(v_cache, desc, &vmap, fp8 ? kMapBlockRows : kMapTileGroups);
            if (st != PKV_OK) return st;
            st = q_map(q, num_seqs, desc, G, QT, &qmap);
            if (st != PKV_OK) return st;
            a.fp8 = fp8 ? 1 : 0;
            cudaError_t e = pkv::launch_prefill_tc(a, qmap, kmap, vmap, s);
            if (e != cudaSuccess) return cuda_fail(e, "cascade prefix launch");
            prefix_launched = true;
        }
    }
    // part 1: each sequence over its own suffix
    {
        int chunk = 0, splits = 0;
        st = plan_decode(desc, num_seqs, max_suffix_len, window, sms, 0, &chunk, &splits);
        if (st != PKV_OK) return st;
        const DecodeWs dws = decode_ws_layout(desc, num_seqs, splits);
        CUtensorMap kmap, vmap;
        st = pool_map(k_cache, desc, &kmap, kMapTileRows);
        if (st != PKV_OK) return st;
        st = pool_map(v_cache, desc, &vmap, kMapTileRows);
        if (st != PKV_OK) return st;
        uint8_t* dwb = wsb + ws.dec;
        pkv::DecodeArgs a{};
        a.q = q;
        a.out = nullptr;
        a.out_f32 = o_parts + rows * desc->head_dim;
        a.lse_out = lse_parts + rows;
        a.block_tables = suffix_tables;
        a.context_lens = suffix_lens;
        a.k_scale = k_scale;
        a.v_scale = v_scale;
        a.counters = dws.total ? reinterpret_cast<uint32_t*>(dwb + dws.counters) : nullptr;
        a.part_lse = dws.total ? reinterpret_cast<float*>(dwb + dws.lse) : nullptr;
        a.part_o = dws.total ? reinterpret_cast<float*>(dwb + dws.o) : nullptr;
        a.err = err;
        a.num_seqs = num_seqs;
        a.hq = desc->num_q_heads;
        a.hkv = desc->num_kv_heads;
        a.group = G;
        a.d = desc->head_dim;
        a.mbps = desc->max_blocks_per_seq;
        a.window = window;
        a.chunk_blocks = chunk;
        a.max_splits = splits;
        a.max_ctx = max_suffix_len;
        a.fp8 = fp8 ? 1 : 0;
        a.num_blocks = desc->num_blocks;
        a.sm_scale = sm_scale;
        // the suffix pass reads nothing the prefix pass writes: it runs under
        // the prefix pass's tail and waits for it only before exiting (the
        // prefix kernel itself waited for everything before it in the stream)
        a.defer_wait = prefix_launched ? 1 : 0;
        cudaError_t e = pkv::launch_decode(a, kmap, vmap, s);
        if (e != cudaSuccess) return cuda_fail(e, "cascade suffix launch");
    }
    // the two states, merged per (sequence, head); without a prefix pass the
    // suffix state alone
    pkv::MergeArgs m{prefix_launched ? o_parts : o_parts + rows * desc->head_dim,
                     prefix_launched ? lse_parts : lse_parts + rows, out, lse_out, prefix_launched ? 2 : 1,
                     num_seqs, desc->num_q_heads, desc->head_dim};
    cudaError_t e = pkv::launch_merge(m, s);
    if (e != cudaSuccess) return cuda_fail(e, "cascade merge launch");
    return PKV_OK;
}

pkv_status pkv_test_inject_wait_timeout(int32_t kernels, uint32_t limit_us) {
    g_last_error[0] = 0;
    if (kernels < 0 || kernels > 3) return fail(PKV_ERR_INVALID_ARG, "kernels mask %d outside [0, 3]", kernels);
    if (kernels && (limit_us < 1 || limit_us > 1000000))
        return fail(PKV_ERR_INVALID_ARG, "limit_us %u outside [1, 1000000]", limit_us);
    g_inject_limit_us.store(limit_us);
    g_inject_kernels.store(kernels);
    return PKV_OK;
}

pkv_status pkv_device_errors(uint32_t* flags_out, int32_t reset) {
    g_last_error[0] = 0;
    if (!flags_out) return fail(PKV_ERR_INVALID_ARG, "flags_out is NULL");
    uint32_t* err = nullptr;
    pkv_status st = device_state(&err, nullptr);
    if (st != PKV_OK) return st;
    cudaError_t e = cudaMemcpyFromSymbol(flags_out, g_pkv_device_error, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (reset) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_pkv_device_error, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "reset device error word");
    }
    return PKV_OK;
}

}  // extern "C"

// ============================================ decode without allocation ==
//
// Some callers cannot allocate device memory when they call in: code that
// runs where cudaMalloc is forbidden or unsafe (inside a custom allocator's
// own callbacks, in a process whose memory pool is locked by its framework,
// or in a plugin that is handed only the tensors it reads and writes), so
// they cannot provide the decode workspace.  This entry point uses a fixed
// scratch array that lives in the library's own device memory instead.

// Fixed scratch for pkv_decode_attention_static: 16 MiB, 256-byte aligned.
// Every GPU that loads the library holds one copy of it until the process
// exits.  Every call shares it and it keeps the last call's contents.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_pkv_static_scratch[kStaticScratchBytes];

namespace {

std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  In host code the array's name is
// only a host-side stand-in, so the address must come from the runtime.
pkv_status static_scratch(void** out, size_t* bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pkv_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode scratch)");
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    *bytes = kStaticScratchBytes;
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_static(
    const pkv_cache_desc* desc, const void* q, const void* k_cache, const void* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len, float sm_scale,
    int32_t window, const float* sinks, int32_t chunk_blocks, void* out, float* lse_out,
    pkv_stream_t stream) {
    return decode_impl(desc, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                       max_context_len, sm_scale, window, sinks, chunk_blocks, out, lse_out, nullptr, 0,
                       stream, nullptr, Scratch::kStatic);
}
