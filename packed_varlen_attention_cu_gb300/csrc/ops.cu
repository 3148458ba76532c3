// ops.cu -- memory-bound companions of the attention kernel:
//   merge of two partial (O, LSE) results (online-softmax combine),
//   zigzag shard index maps, and row gather/scatter.
//
// "03 · 长文负载均衡" §3.2 (DCP): partial outputs of several computation blocks
// of one O block are reduced by online-softmax rescale-and-sum; the ring
// attention loop of "长序列训练与上下文并行" merges each step's local result
// into the running state.  §4.2-4.3: zigzag (rank i owns chunks i and
// 2cp-1-i) applied to every document on its own.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pva.h"
#include "common.h"

namespace pva {
namespace {

int grid_for(int64_t work_items, int threads) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 16;  // grid-stride beyond 16 waves of CTAs
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// ------------------------------------------------------------------ merge
// Each (token, head) row of O is cpr = d / kElems 16-byte chunks; a warp
// covers 32 / cpr whole rows (the host accepts only head dims whose chunk
// count divides 32).  Per row, the lane holding chunk 0 loads the two LSEs and
// computes the weights once; the row's other lanes receive them by shuffle.
// Each thread handles kMergeUnroll chunks per pass (whole warps at a stride of
// the grid), all loads issued before any arithmetic, so that enough bytes are
// in flight to keep HBM busy.
constexpr int kMergeThreads = 256;
// chunks per thread and pass: measured over a 131072 x 32 x 128 fp32 merge on
// GB300 (in place / out of place, GB/s): 1: 5681 / 6472, 2: 5652 / 6288,
// 3: 5920 / 6687, 4: 5400 / 5990, 8: 3014 / 3045
constexpr int kMergeUnroll = 3;

template <bool F32>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(
    const void* __restrict__ oa_, const float* la, const void* __restrict__ ob_, const float* lb,
    void* out_, float* lout, int64_t tokens, int32_t heads, int32_t d) {
    constexpr int kElems = F32 ? 4 : 8;
    const int32_t cpr = d / kElems;  // chunks per row
    const int64_t nchunks = tokens * heads * cpr;
    const int lane = threadIdx.x & 31;
    const int lead = lane & ~(cpr - 1);  // lane of chunk 0 of this lane's row
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const uint4* oa = reinterpret_cast<const uint4*>(oa_);
    const uint4* ob = reinterpret_cast<const uint4*>(ob_);
    uint4* out = reinterpret_cast<uint4*>(out_);
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x - lane; base < nchunks;
         base += kMergeUnroll * stride) {
        uint4 x[kMergeUnroll], y[kMergeUnroll];
        float a[kMergeUnroll], b[kMergeUnroll];
        int64_t li[kMergeUnroll];
#pragma unroll
        for (int u = 0; u < kMergeUnroll; ++u) {
            const int64_t idx = base + u * stride + lane;
            const bool act = idx < nchunks;
            const int64_t row = idx / cpr;
            const int64_t t = row / heads;
            li[u] = (int64_t)(row - t * heads) * tokens + t;
            a[u] = b[u] = -INFINITY;
            if (act && lane == lead) {
                a[u] = la[li[u]];
                b[u] = lb[li[u]];
            }
            if (act) {
                x[u] = oa[idx];
                y[u] = ob[idx];
            }
        }
#pragma unroll
        for (int u = 0; u < kMergeUnroll; ++u) {
            const int64_t idx = base + u * stride + lane;
            const bool act = idx < nchunks;
            float wa = 0.f, wb = 0.f, l = -INFINITY;
            if (lane == lead && (a[u] != -INFINITY || b[u] != -INFINITY)) {
                //   l = ln(e^a + e^b),  w_a = e^(a - l),  w_b = e^(b - l)
                const float mx = fmaxf(a[u], b[u]);
                const float ea = expf(a[u] - mx), eb = expf(b[u] - mx);
                const float inv = 1.f / (ea + eb);
                l = mx + logf(ea + eb);
                wa = ea * inv;
                wb = eb * inv;
            }
            wa = __shfl_sync(0xffffffffu, wa, lead);
            wb = __shfl_sync(0xffffffffu, wb, lead);
            if (!act) continue;
            if (F32) {
                const float4 fx = *reinterpret_cast<const float4*>(&x[u]);
                const float4 fy = *reinterpret_cast<const float4*>(&y[u]);
                const float4 o = make_float4(wa * fx.x + wb * fy.x, wa * fx.y + wb * fy.y,
                                             wa * fx.z + wb * fy.z, wa * fx.w + wb * fy.w);
                out[idx] = *reinterpret_cast<const uint4*>(&o);
            } else {
                const uint32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                const uint32_t ys[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
                uint32_t r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fx =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
                    const float2 fy =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
                    const __nv_bfloat162 o =
                        __floats2bfloat162_rn(wa * fx.x + wb * fy.x, wa * fx.y + wb * fy.y);
                    r[e] = *reinterpret_cast<const uint32_t*>(&o);
                }
                out[idx] = make_uint4(r[0], r[1], r[2], r[3]);
            }
            // the lead lane read the input LSEs itself, so the (possibly in-place)
            // output LSE may be written now
            if (lane == lead) lout[li[u]] = l;
        }
    }
}

// ------------------------------------------------------------------ zigzag
__device__ __forceinline__ void zz_chunk(int32_t len, int32_t cp, int32_t c, int32_t& off,
                                         int32_t& clen) {
    const int32_t n = 2 * cp, base = len / n, rem = len % n;
    clen = base + (c < rem ? 1 : 0);
    off = c * base + (c < rem ? c : rem);
}

constexpr int kZzThreads = 1024;

// One CTA: for each rank of [rank_begin, rank_end), per-document rank-local
// offsets in shared memory (block scan), then every local row is mapped to its
// global token; the ranks' shards follow each other in `map`.
__global__ void __launch_bounds__(kZzThreads) zigzag_kernel(const int32_t* cu, int32_t nd,
                                                             int32_t cp, int32_t rank_begin,
                                                             int32_t rank_end, int32_t* map,
                                                             int32_t* table) {
    extern __shared__ int32_t loc[];  // [nd + 1]
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int32_t row0 = 0;  // first map entry of the current rank
    for (int32_t rank = rank_begin; rank < rank_end; ++rank) {
        if (tid == 0) carry = 0;
        __syncthreads();
        const int32_t c0 = rank, c1 = 2 * cp - 1 - rank;
        for (int32_t d0 = 0; d0 < nd; d0 += kZzThreads) {
            const int32_t d = d0 + tid;
            int32_t v = 0;
            if (d < nd) {
                const int32_t len = cu[d + 1] - cu[d];
                int32_t o0, l0, o1, l1;
                zz_chunk(len, cp, c0, o0, l0);
                zz_chunk(len, cp, c1, o1, l1);
                v = l0 + l1;
                if (table) {
                    int32_t* r = table + (int64_t)d * 8;
                    r[0] = d; r[1] = c0; r[2] = cu[d] + o0; r[3] = l0;
                    r[4] = d; r[5] = c1; r[6] = cu[d] + o1; r[7] = l1;
                }
            }
            int32_t inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += t;
            }
            if (lane == 31) warp_sum[w] = inc;
            __syncthreads();
            if (w == 0) {
                int32_t x = warp_sum[lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t t = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += t;
                }
                warp_sum[lane] = x;
            }
            __syncthreads();
            if (d < nd) loc[d] = carry + (w > 0 ? warp_sum[w - 1] : 0) + inc - v;
            __syncthreads();
            if (tid == 0) carry += warp_sum[31];
            __syncthreads();
        }
        if (tid == 0) loc[nd] = carry;
        __syncthreads();
        const int32_t total = loc[nd];
        for (int32_t i = tid; i < total; i += kZzThreads) {
            int32_t lo = 0, hi = nd - 1;  // last document with loc[d] <= i
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if (loc[mid] <= i) lo = mid;
                else hi = mid - 1;
            }
            const int32_t d = lo, len = cu[d + 1] - cu[d], j = i - loc[d];
            int32_t o0, l0, o1, l1;
            zz_chunk(len, cp, c0, o0, l0);
            zz_chunk(len, cp, c1, o1, l1);
            map[row0 + i] = cu[d] + (j < l0 ? o0 + j : o1 + (j - l0));
        }
        row0 += total;
        __syncthreads();  // loc[] is rewritten for the next rank
    }
}

// ------------------------------------------------------------------ gather
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ src,
                                                     const int32_t* __restrict__ map,
                                                     uint4* __restrict__ dst, int64_t rows,
                                                     int64_t chunks_per_row, int64_t indexed_rows,
                                                     int32_t scatter) {
    const int64_t n = rows * chunks_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += stride) {
        const int64_t r = idx / chunks_per_row, c = idx - r * chunks_per_row;
        const int64_t m = map[r];
        if (m < 0 || m >= indexed_rows) continue;
        if (scatter) dst[m * chunks_per_row + c] = src[idx];
        else dst[idx] = src[m * chunks_per_row + c];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pva

using namespace pva;

extern "C" pva_status pva_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                                         const float* lse_b, void* out, float* lse_out,
                                         int64_t tokens, int32_t heads, int32_t head_dim,
                                         int32_t o_is_fp32, void* stream) {
    if (tokens < 0 || heads <= 0 || (o_is_fp32 != 0 && o_is_fp32 != 1)) return PVA_ERR_INVALID_ARG;
    // a row's 16-byte chunks must divide a warp (in-place LSE update, see kernel)
    const int32_t cpr = head_dim / (o_is_fp32 ? 4 : 8);
    if (head_dim <= 0 || head_dim % (o_is_fp32 ? 4 : 8) != 0 || cpr > 32 || 32 % cpr != 0)
        return PVA_ERR_UNSUPPORTED;
    if (tokens == 0) return PVA_OK;
    if (!o_a || !o_b || !out || !lse_a || !lse_b || !lse_out) return PVA_ERR_INVALID_ARG;
    if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(out) || !aligned16(lse_a) ||
        !aligned16(lse_b) || !aligned16(lse_out))
        return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t chunks = tokens * heads * (head_dim / (o_is_fp32 ? 4 : 8));
    const int grid = grid_for((chunks + kMergeUnroll - 1) / kMergeUnroll, kMergeThreads);
    if (o_is_fp32)
        merge_kernel<true><<<grid, kMergeThreads, 0, st>>>(o_a, lse_a, o_b, lse_b, out, lse_out,
                                                           tokens, heads, head_dim);
    else
        merge_kernel<false><<<grid, kMergeThreads, 0, st>>>(o_a, lse_a, o_b, lse_b, out, lse_out,
                                                            tokens, heads, head_dim);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" pva_status pva_zigzag_shard(const int32_t* cu_seqlens_dev, int32_t num_docs, int32_t cp,
                                       int32_t rank, int32_t* gather_map_dev,
                                       int32_t* chunk_table_dev, void* stream) {
    if (!cu_seqlens_dev || !gather_map_dev || num_docs < 0 || cp < 1 || rank < 0 || rank >= cp)
        return PVA_ERR_INVALID_ARG;
    const size_t smem = ((size_t)num_docs + 1) * sizeof(int32_t);
    if (smem > 200 * 1024) return PVA_ERR_UNSUPPORTED;  // more than ~51K documents
    if (num_docs == 0) return PVA_OK;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(zigzag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return PVA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    zigzag_kernel<<<1, kZzThreads, smem, st>>>(cu_seqlens_dev, num_docs, cp, rank, rank + 1,
                                               gather_map_dev, chunk_table_dev);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" pva_status pva_zigzag_ring_map(const int32_t* cu_seqlens_dev, int32_t num_docs,
                                          int32_t cp, int32_t* ring_map_dev, void* stream) {
    if (!cu_seqlens_dev || !ring_map_dev || num_docs < 0 || cp < 1) return PVA_ERR_INVALID_ARG;
    const size_t smem = ((size_t)num_docs + 1) * sizeof(int32_t);
    if (smem > 200 * 1024) return PVA_ERR_UNSUPPORTED;
    if (num_docs == 0) return PVA_OK;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(zigzag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return PVA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    zigzag_kernel<<<1, kZzThreads, smem, st>>>(cu_seqlens_dev, num_docs, cp, 0, cp, ring_map_dev,
                                               nullptr);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" pva_status pva_gather_rows(const void* src, const int32_t* map_dev, void* dst,
                                      int64_t rows, int64_t row_bytes, int64_t indexed_rows,
                                      int32_t scatter, void* stream) {
    if (rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0 || indexed_rows < 0 ||
        (scatter != 0 && scatter != 1))
        return PVA_ERR_INVALID_ARG;
    if (rows == 0) return PVA_OK;
    if (!src || !dst || !map_dev || !aligned16(src) || !aligned16(dst)) return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t cpr = row_bytes / 16;
    gather_kernel<<<grid_for(rows * cpr, 256), 256, 0, st>>>(
        reinterpret_cast<const uint4*>(src), map_dev, reinterpret_cast<uint4*>(dst), rows, cpr,
        indexed_rows, scatter);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}
