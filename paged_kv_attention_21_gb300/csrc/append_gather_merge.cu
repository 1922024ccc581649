// append_gather_merge.cu -- the small kernels of the path:
//   * fused KV append + RoPE (+ e4m3 quantisation)  (llm-infer, "What It Does":
//     KV writes and fused RoPE inside the decode step);
//   * block-table gather of one pool into contiguous rows (infer-lab,
//     "Technique" table: PagedAttention block tables);
//   * copy-on-write of whole blocks (infer-lab, "Technique" table:
//     refcounting, copy-on-write; llm-infer, "What It Does");
//   * standalone merge of partial (o, lse) states (FlashAttention-2 work
//     partitioning, cited under llm-infer "References").
// All of them are latency-bound: a few MB at most.  Loads and stores are
// coalesced across the warp; no shared memory is needed.
#include "common.cuh"
#include "internal.h"

namespace pkv {

// ------------------------------------------------------- append + RoPE --
//
// One warp per (token, row), rows = the Hkv KV heads (K and V together)
// followed by the Hq query heads.  Lane l owns the rotation pairs
// (j, j + D/2) for j in [l*PPL, (l+1)*PPL).

template <int D, bool kFp8>
__global__ void __launch_bounds__(256) append_rope_kernel(AppendArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int HALF = D / 2;
    constexpr int PPL = HALF / 32;  // 1 for D=64, 2 for D=128
    const int lane = threadIdx.x & 31;
    const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int rows = a.hkv + ((a.q != nullptr && a.cos_sin != nullptr) ? a.hq : 0);
    const long long i = w / rows;
    const int r = static_cast<int>(w % rows);
    if (i >= a.num_tokens) return;

    const int s = a.token_to_seq[i];
    const int p = a.positions[i];
    const int tb = a.ring > 0 ? (p / kBlockSize) % a.ring : p / kBlockSize;  // table entry
    const bool ok = s >= 0 && s < a.num_seqs && p >= 0 && tb < a.mbps &&
                    (a.cos_sin == nullptr || p < a.max_pos);
    if (!ok) {
        if (lane == 0) flag_error(a.err, PKV_DEVERR_POSITION);
        return;
    }
    const int j0 = lane * PPL;
    float c[PPL], sn[PPL];
    const bool rope = a.cos_sin != nullptr;
    if (rope) {
        const float* cs = a.cos_sin + (static_cast<size_t>(p) * HALF + j0) * 2;
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            c[k] = cs[2 * k];
            sn[k] = cs[2 * k + 1];
        }
    }

    // Load this lane's pairs of a bf16 row and (optionally) rotate them.
    auto rotate = [&](const __nv_bfloat16* x, float (&lo)[PPL], float (&hi)[PPL]) {
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            const float av = __bfloat162float(x[j0 + k]);
            const float bv = __bfloat162float(x[HALF + j0 + k]);
            if (rope) {
                // x'[j] = a*c - b*s ; x'[j+D/2] = b*c + a*s ; each op rounded
                lo[k] = __fsub_rn(__fmul_rn(av, c[k]), __fmul_rn(bv, sn[k]));
                hi[k] = __fadd_rn(__fmul_rn(bv, c[k]), __fmul_rn(av, sn[k]));
            } else {
                lo[k] = av;
                hi[k] = bv;
            }
        }
    };

    if (r < a.hkv) {
        const int blk = a.block_tables[static_cast<size_t>(s) * a.mbps + tb];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
            return;
        }
        const size_t src = (static_cast<size_t>(i) * a.hkv + r) * D;
        const size_t dst = ((static_cast<size_t>(blk) * a.hkv + r) * kBlockSize + p % kBlockSize) * D;
        const __nv_bfloat16* kx = static_cast<const __nv_bfloat16*>(a.k_new) + src;
        const __nv_bfloat16* vx = static_cast<const __nv_bfloat16*>(a.v_new) + src;
        float lo[PPL], hi[PPL];
        rotate(kx, lo, hi);
        if constexpr (!kFp8) {
            __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(a.k_cache) + dst;
            __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(a.v_cache) + dst;
#pragma unroll
            for (int k = 0; k < PPL; ++k) {
                kc[j0 + k] = __float2bfloat16_rn(lo[k]);
                kc[HALF + j0 + k] = __float2bfloat16_rn(hi[k]);
                vc[j0 + k] = vx[j0 + k];
                vc[HALF + j0 + k] = vx[HALF + j0 + k];
            }
        } else {
            uint8_t* kc = static_cast<uint8_t*>(a.k_cache) + dst;
            uint8_t* vc = static_cast<uint8_t*>(a.v_cache) + dst;
            const float ks = a.k_scale[r];
            const float vs = a.v_scale[r];
#pragma unroll
            for (int k = 0; k < PPL; ++k) {
                kc[j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(lo[k], ks), __NV_SATFINITE, __NV_E4M3);
                kc[HALF + j0 + k] =
                    __nv_cvt_float_to_fp8(__fdiv_rn(hi[k], ks), __NV_SATFINITE, __NV_E4M3);
                vc[j0 + k] = __nv_cvt_float_to_fp8(__fdiv_rn(__bfloat162float(vx[j0 + k]), vs),
                                                   __NV_SATFINITE, __NV_E4M3);
                vc[HALF + j0 + k] =
                    __nv_cvt_float_to_fp8(__fdiv_rn(__bfloat162float(vx[HALF + j0 + k]), vs),
                                          __NV_SATFINITE, __NV_E4M3);
            }
        }
    } else {
        const int h = r - a.hkv;
        __nv_bfloat16* qx = static_cast<__nv_bfloat16*>(a.q) + (static_cast<size_t>(i) * a.hq + h) * D;
        float lo[PPL], hi[PPL];
        rotate(qx, lo, hi);
        __syncwarp();  // every lane has read its pairs before any lane writes
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            qx[j0 + k] = __float2bfloat16_rn(lo[k]);
            qx[HALF + j0 + k] = __float2bfloat16_rn(hi[k]);
        }
    }
}

cudaError_t launch_append_rope(const AppendArgs& a, cudaStream_t stream) {
    const int rows = a.hkv + ((a.q != nullptr && a.cos_sin != nullptr) ? a.hq : 0);
    const long long warps = static_cast<long long>(a.num_tokens) * rows;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(blocks));
    cudaError_t e;
    if (a.d == 64) {
        if (a.fp8) e = launch_pdl(append_rope_kernel<64, true>, grid, dim3(threads), 0, stream, a);
        else e = launch_pdl(append_rope_kernel<64, false>, grid, dim3(threads), 0, stream, a);
    } else {
        if (a.fp8) e = launch_pdl(append_rope_kernel<128, true>, grid, dim3(threads), 0, stream, a);
        else e = launch_pdl(append_rope_kernel<128, false>, grid, dim3(threads), 0, stream, a);
    }
    return e;
}

// --------------------------------------------------------------- gather --
//
// One thread per 16-byte chunk of an output row.

__global__ void __launch_bounds__(256) gather_kernel(GatherArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int chunks = a.row_bytes / 16;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long per_token = static_cast<long long>(a.hkv) * chunks;
    const long long g = idx / per_token;
    if (g >= a.total_tokens) return;
    const int h = static_cast<int>((idx / chunks) % a.hkv);
    const int c = static_cast<int>(idx % chunks);
    // sequence owning output row g: last s with cu_lens[s] <= g
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu_lens[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    const int t = static_cast<int>(g - a.cu_lens[s]);
    if (t < 0 || t >= a.lens[s] || t / kBlockSize >= a.mbps) {
        if (c == 0 && h == 0) flag_error(a.err, PKV_DEVERR_POSITION);
        return;
    }
    const int blk = a.block_tables[static_cast<size_t>(s) * a.mbps + t / kBlockSize];
    if (blk < 0 || blk >= a.num_blocks) {
        if (c == 0 && h == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const uint8_t*>(a.cache) +
        ((static_cast<size_t>(blk) * a.hkv + h) * kBlockSize + t % kBlockSize) * a.row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                          (static_cast<size_t>(g) * a.hkv + h) * a.row_bytes);
    dst[c] = src[c];
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream) {
    const long long n = a.total_tokens * a.hkv * (a.row_bytes / 16);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (n + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    return launch_pdl(gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, a);
}

// ----------------------------------------------------------- block copy --
//
// Copy-on-write: one CTA per (pair, pool); 16-byte vector copies of the
// whole block (every head and row).

__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int i = blockIdx.x;
    const int src = a.src[i];
    const int dst = a.dst[i];
    if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
        if (threadIdx.x == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    uint8_t* pool = static_cast<uint8_t*>(blockIdx.y == 0 ? a.k_cache : a.v_cache);
    const uint4* s = reinterpret_cast<const uint4*>(pool + static_cast<size_t>(src) * a.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(pool + static_cast<size_t>(dst) * a.block_bytes);
    const int n = static_cast<int>(a.block_bytes / 16);
    for (int c = threadIdx.x; c < n; c += blockDim.x) d[c] = s[c];
}

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream) {
    if (a.num_pairs == 0) return cudaSuccess;
    return launch_pdl(copy_blocks_kernel, dim3(a.num_pairs, 2), dim3(256), 0, stream, a);
}

// ---------------------------------------------------------------- merge --
//
// One warp per (row, head); lanes stride over head_dim.
//   M = max_i lse_i ; w_i = exp(lse_i - M) ; o = sum w_i o_i / sum w_i ;
//   lse = M + ln sum w_i.   Empty parts (lse = -inf) are skipped.

__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long RH = static_cast<long long>(a.num_rows) * a.num_heads;
    if (w >= RH) return;
    float M = -INFINITY;
    for (int i = 0; i < a.num_parts; ++i) M = fmaxf(M, a.lse_parts[i * RH + w]);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + w * a.head_dim;
    if (M == -INFINITY) {
        for (int d = lane; d < a.head_dim; d += 32) out[d] = __float2bfloat16_rn(0.0f);
        if (a.lse_out && lane == 0) a.lse_out[w] = -INFINITY;
        return;
    }
    float W = 0.0f;
    for (int i = 0; i < a.num_parts; ++i) {
        const float l = a.lse_parts[i * RH + w];
        if (l != -INFINITY) W += expf(l - M);
    }
    const float invW = 1.0f / W;
    for (int d = lane; d < a.head_dim; d += 32) {
        float acc = 0.0f;
        for (int i = 0; i < a.num_parts; ++i) {
            const float l = a.lse_parts[i * RH + w];
            if (l == -INFINITY) continue;
            acc += expf(l - M) * a.o_parts[(i * RH + w) * a.head_dim + d];
        }
        out[d] = __float2bfloat16_rn(acc * invW);
    }
    if (a.lse_out && lane == 0) a.lse_out[w] = M + logf(W);
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    const long long warps = static_cast<long long>(a.num_rows) * a.num_heads;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    return launch_pdl(merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, a);
}

}  // namespace pkv

namespace pkv {

// ------------------------------------------------- ring-cache prefill --
//
// Staging: one warp per (sequence, staging block, head, row); lane l moves
// D/32 elements of the K row and of the V row.  Position p = start + 16 b +
// row comes from the ring below the chunk, from the chunk's own K/V inside
// it (e4m3 rings: quantised as the append quantises, then widened), and is
// zero past kv_len.

__device__ __forceinline__ int ring_start(int kv_len, int q_len, int window) {
    const int lo = max(0, kv_len - q_len - window + 1);
    return lo - lo % kBlockSize;
}

__device__ __forceinline__ uint16_t bf16_bits_of(float x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&b);
}

__device__ __forceinline__ float e4m3_value(uint8_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
    return __half2float(__half(h));
}

template <int D>
__global__ void __launch_bounds__(256) stage_ring_kernel(RingStageArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int EPL = D / 32;  // elements per lane
    const int lane = threadIdx.x & 31;
    const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long per_seq = static_cast<long long>(a.cap) * a.hkv * kBlockSize;
    const int s = static_cast<int>(w / per_seq);
    if (s >= a.num_seqs) return;
    const long long rem = w % per_seq;
    const int b = static_cast<int>(rem / (a.hkv * kBlockSize));
    const int h = static_cast<int>((rem / kBlockSize) % a.hkv);
    const int row = static_cast<int>(rem % kBlockSize);
    const int q0 = a.qo_indptr[s];
    const int q_len = a.qo_indptr[s + 1] - q0;
    const int kv_len = a.kv_lens[s];
    const int start = ring_start(kv_len, q_len, a.window);
    const int prefix = kv_len - q_len;
    if (lane == 0 && h == 0 && row == 0) {
        a.stage_tables[static_cast<size_t>(s) * a.cap + b] = s * a.cap + b;
        if (b == 0) a.stage_lens[s] = kv_len - start;
    }
    const int p = start + b * kBlockSize + row;
    const size_t dst = ((static_cast<size_t>(s) * a.cap + b) * a.hkv + h) * kBlockSize * D + row * D;
    uint16_t kv[2][EPL];
    if (p < prefix && p >= 0) {
        const int entry = (p / kBlockSize) % a.ring;
        const int blk = a.block_tables[static_cast<size_t>(s) * a.mbps + entry];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
#pragma unroll
            for (int e = 0; e < EPL; ++e) kv[0][e] = kv[1][e] = 0;
        } else {
            const size_t src = ((static_cast<size_t>(blk) * a.hkv + h) * kBlockSize + p % kBlockSize) * D;
#pragma unroll
            for (int pool = 0; pool < 2; ++pool) {
                const void* base = pool ? a.v_cache : a.k_cache;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const int c = lane + 32 * e;
                    kv[pool][e] = a.fp8 ? bf16_bits_of(e4m3_value(static_cast<const uint8_t*>(base)[src + c]))
                                        : static_cast<const uint16_t*>(base)[src + c];
                }
            }
        }
    } else if (p >= prefix && p < kv_len) {
        const size_t src = (static_cast<size_t>(q0 + p - prefix) * a.hkv + h) * D;
#pragma unroll
        for (int pool = 0; pool < 2; ++pool) {
            const uint16_t* x = static_cast<const uint16_t*>(pool ? a.v_chunk : a.k_chunk) + src;
            const float sc = a.fp8 ? (pool ? a.v_scale[h] : a.k_scale[h]) : 1.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const uint16_t v = x[lane + 32 * e];
                if (a.fp8) {
                    const float f = __uint_as_float(static_cast<uint32_t>(v) << 16);
                    const uint8_t code = __nv_cvt_float_to_fp8(__fdiv_rn(f, sc), __NV_SATFINITE, __NV_E4M3);
                    kv[pool][e] = bf16_bits_of(e4m3_value(code));
                } else {
                    kv[pool][e] = v;
                }
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) kv[0][e] = kv[1][e] = 0;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        a.k_stage[dst + lane + 32 * e] = kv[0][e];
        a.v_stage[dst + lane + 32 * e] = kv[1][e];
    }
}

// Commit: one warp per (chunk token, head); the tokens at positions >=
// kv_len - ring * 16 (the ones the ring keeps, each in its own slot) are
// written into the ring as the append writes them (K already rotated).
template <int D>
__global__ void __launch_bounds__(256) commit_ring_kernel(RingStageArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int EPL = D / 32;
    const int lane = threadIdx.x & 31;
    const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long t = w / a.hkv;
    const int h = static_cast<int>(w % a.hkv);
    if (t >= a.total_q) return;
    // the sequence of chunk row t: the last s with qo_indptr[s] <= t
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.qo_indptr[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int q0 = a.qo_indptr[s];
    const int q_len = a.qo_indptr[s + 1] - q0;
    if (t >= q0 + q_len) return;  // a row past the batch's last sequence
    const int kv_len = a.kv_lens[s];
    const int p = kv_len - q_len + static_cast<int>(t - q0);
    if (p < 0 || p < kv_len - a.ring * kBlockSize) return;  // overwritten within this chunk
    const int entry = (p / kBlockSize) % a.ring;
    const int blk = a.block_tables[static_cast<size_t>(s) * a.mbps + entry];
    if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) flag_error(a.err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    const size_t src = (static_cast<size_t>(t) * a.hkv + h) * D;
    const size_t dst = ((static_cast<size_t>(blk) * a.hkv + h) * kBlockSize + p % kBlockSize) * D;
#pragma unroll
    for (int pool = 0; pool < 2; ++pool) {
        const uint16_t* x = static_cast<const uint16_t*>(pool ? a.v_chunk : a.k_chunk) + src;
        if (a.fp8) {
            uint8_t* c = static_cast<uint8_t*>(pool ? a.v_ring_out : a.k_ring_out) + dst;
            const float sc = pool ? a.v_scale[h] : a.k_scale[h];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const float f = __uint_as_float(static_cast<uint32_t>(x[lane + 32 * e]) << 16);
                c[lane + 32 * e] = __nv_cvt_float_to_fp8(__fdiv_rn(f, sc), __NV_SATFINITE, __NV_E4M3);
            }
        } else {
            uint16_t* c = static_cast<uint16_t*>(pool ? a.v_ring_out : a.k_ring_out) + dst;
#pragma unroll
            for (int e = 0; e < EPL; ++e) c[lane + 32 * e] = x[lane + 32 * e];
        }
    }
}

cudaError_t launch_stage_ring(const RingStageArgs& a, cudaStream_t stream) {
    const long long warps = static_cast<long long>(a.num_seqs) * a.cap * a.hkv * kBlockSize;
    if (warps == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
    return a.d == 64 ? launch_pdl(stage_ring_kernel<64>, grid, dim3(256), 0, stream, a)
                     : launch_pdl(stage_ring_kernel<128>, grid, dim3(256), 0, stream, a);
}

cudaError_t launch_commit_ring(const RingStageArgs& a, cudaStream_t stream) {
    const long long warps = static_cast<long long>(a.total_q) * a.hkv;
    if (warps == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((warps + 7) / 8));
    return a.d == 64 ? launch_pdl(commit_ring_kernel<64>, grid, dim3(256), 0, stream, a)
                     : launch_pdl(commit_ring_kernel<128>, grid, dim3(256), 0, stream, a);
}

}  // namespace pkv
