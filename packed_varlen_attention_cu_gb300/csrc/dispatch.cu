// dispatch.cu -- sharding solvers for context parallelism on the worklist's
// cost code ("03 · 长文负载均衡" §4.2-§4.4):
//   chunk mask areas and the greedy min-heap dispatch of MagiAttention (§4.4),
//   striped shard maps (§4.2), and WLB-LLM's per-sequence vs per-document
//   choice on tile-rounded FLOPs (§4.3).
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <vector>

#include "../../include/pva.h"

namespace pva {
namespace {

constexpr int kAreaThreads = 256;
constexpr int kDispatchThreads = 1024;
constexpr int32_t kMaxDispatchChunks = 8192;
constexpr int32_t kMaxDispatchBuckets = 1024;

// Allowed keys of packed query row i: its document's causal prefix (bounded by
// the window), plus every question token for an answer row of a shared
// question mask.  Rows past cu[ndocs] have none.
__device__ __forceinline__ int64_t row_area(const int32_t* cu, int32_t ndocs, int32_t kind,
                                            int32_t window, int32_t nprefix, int32_t i) {
    int32_t lo = 0, hi = ndocs;  // last d with cu[d] <= i
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= i) lo = mid;
        else hi = mid - 1;
    }
    const int32_t d = lo;
    if (d >= ndocs || i >= cu[d + 1]) return 0;
    const int64_t pos = i - cu[d];
    switch (kind) {
    case PVA_MASK_SLIDING_WINDOW:
        return pos + 1 < window ? pos + 1 : window;
    case PVA_MASK_SHARED_QUESTION:
        return d < nprefix ? pos + 1 : (int64_t)cu[nprefix] + pos + 1;
    default:
        return pos + 1;
    }
}

// One CTA per chunk of chunk_size query rows: the chunk's allowed pairs.
__global__ void __launch_bounds__(kAreaThreads)
    chunk_area_kernel(const int32_t* cu, int32_t ndocs, int32_t kind, int32_t window,
                      int32_t nprefix, int32_t T, int32_t chunk_size, int64_t* areas) {
    __shared__ unsigned long long part[kAreaThreads / 32];
    const int64_t r0 = (int64_t)blockIdx.x * chunk_size;
    const int64_t r1 = r0 + chunk_size < T ? r0 + chunk_size : T;
    unsigned long long s = 0;
    for (int64_t i = r0 + threadIdx.x; i < r1; i += kAreaThreads)
        s += (unsigned long long)row_area(cu, ndocs, kind, window, nprefix, (int32_t)i);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < kAreaThreads / 32; ++w) t += part[w];
        areas[blockIdx.x] = (int64_t)t;
    }
}

// Greedy min-heap dispatch, one CTA.  Chunks are sorted by (area desc, index
// asc) with a bitonic sort in shared memory; then one warp walks them in that
// order and gives each to the bucket with the smallest area that still has
// room (ties: lower bucket id), which is the same choice the min-heap of the
// pages makes: a warp arg-min over at most 1024 buckets per chunk.
__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_kernel(const int64_t* areas, int32_t n, int32_t cp, int32_t* bucket,
                    int64_t* loads_out) {
    extern __shared__ unsigned long long dsm[];
    int32_t np2 = 1;
    while (np2 < n) np2 <<= 1;
    long long* a = reinterpret_cast<long long*>(dsm);             // [np2]
    int32_t* idx = reinterpret_cast<int32_t*>(a + np2);           // [np2]
    long long* load = reinterpret_cast<long long*>(idx + np2 + (np2 & 1));  // [cp]
    int32_t* fill = reinterpret_cast<int32_t*>(load + cp);        // [cp]
    for (int32_t i = threadIdx.x; i < np2; i += kDispatchThreads) {
        a[i] = i < n ? areas[i] : -1;  // padding sorts last
        idx[i] = i;
    }
    for (int32_t b = threadIdx.x; b < cp; b += kDispatchThreads) {
        load[b] = 0;
        fill[b] = 0;
    }
    __syncthreads();
    // "x before y": larger area first, then lower index
    for (int32_t size = 2; size <= np2; size <<= 1) {
        for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (int32_t t = threadIdx.x; t < np2 / 2; t += kDispatchThreads) {
                const int32_t lo = 2 * t - (t & (stride - 1));
                const int32_t hi = lo + stride;
                const bool up = (lo & size) == 0;
                const long long xa = a[lo], ya = a[hi];
                const int32_t xi = idx[lo], yi = idx[hi];
                const bool x_first = xa > ya || (xa == ya && xi < yi);
                if (x_first != up) {
                    a[lo] = ya;
                    a[hi] = xa;
                    idx[lo] = yi;
                    idx[hi] = xi;
                }
            }
            __syncthreads();
        }
    }
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int32_t cap = n / cp;
        for (int32_t t = 0; t < n; ++t) {
            long long best = LLONG_MAX;
            int32_t bid = INT32_MAX;
            for (int32_t b = lane; b < cp; b += 32) {
                if (fill[b] < cap && load[b] < best) {  // ascending b: lowest id on ties
                    best = load[b];
                    bid = b;
                }
            }
            for (int o = 16; o > 0; o >>= 1) {
                const long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int32_t oi = __shfl_xor_sync(0xffffffffu, bid, o);
                if (ob < best || (ob == best && oi < bid)) {
                    best = ob;
                    bid = oi;
                }
            }
            if (lane == 0) {
                load[bid] += a[t];
                fill[bid] += 1;
                bucket[idx[t]] = bid;
            }
            __syncwarp();
        }
    }
    __syncthreads();
    for (int32_t b = threadIdx.x; b < cp; b += kDispatchThreads) loads_out[b] = load[b];
}

// Rank `rank`'s tokens under striped sharding, in order: its k-th token is in
// stripe rank + cp * (k / stripe), at offset k % stripe.
__global__ void striped_kernel(int32_t T, int32_t cp, int32_t rank, int32_t stripe, int32_t n,
                               int32_t* map) {
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s = rank + (int64_t)cp * (k / stripe);
        const int64_t tok = s * stripe + k % stripe;
        if (tok < T) map[k] = (int32_t)tok;
    }
}

size_t dispatch_smem(int32_t n, int32_t cp) {
    int32_t np2 = 1;
    while (np2 < n) np2 <<= 1;
    return (size_t)np2 * 8 + (size_t)(np2 + (np2 & 1)) * 4 + (size_t)cp * 12;
}

// Zigzag chunk c of a length-len sequence cut into 2 cp chunks: the first
// len mod 2cp chunks hold one extra token.
void zz_chunk(int32_t len, int32_t cp, int32_t c, int32_t* off, int32_t* clen) {
    const int32_t n = 2 * cp, base = len / n, rem = len % n;
    *clen = base + (c < rem ? 1 : 0);
    *off = c * base + (c < rem ? c : rem);
}

// Tile-rounded causal FLOPs of positions [p0, p1) of one document: q tiles
// aligned at p0, a q tile whose last position is P computes ceil((P+1)/tile)
// key tiles (keys are aligned at the document start).
int64_t piece_flops(int32_t p0, int32_t p1, int32_t tile, int32_t d) {
    int64_t tiles = 0;
    for (int64_t r = p0; r < p1; r += tile) {
        const int64_t last = r + tile < p1 ? r + tile - 1 : p1 - 1;
        tiles += (last + tile) / tile;
    }
    return tiles * tile * tile * 4 * d;
}

}  // namespace
}  // namespace pva

using namespace pva;

extern "C" pva_status pva_chunk_areas(const int32_t* cu_seqlens_dev, int32_t num_docs,
                                      const pva_mask_desc* mask, int32_t chunk_size,
                                      int64_t* areas_dev, void* stream) {
    if (!cu_seqlens_dev || !mask || !areas_dev || num_docs < 0 || chunk_size <= 0)
        return PVA_ERR_INVALID_ARG;
    if (mask->kind != PVA_MASK_CAUSAL && mask->kind != PVA_MASK_SLIDING_WINDOW &&
        mask->kind != PVA_MASK_SHARED_QUESTION)
        return PVA_ERR_UNSUPPORTED;
    if (mask->kind == PVA_MASK_SLIDING_WINDOW && mask->window < 1) return PVA_ERR_INVALID_ARG;
    if (mask->kind == PVA_MASK_SHARED_QUESTION &&
        (mask->num_prefix_docs < 0 || mask->num_prefix_docs > num_docs))
        return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens < 0 || mask->q_tokens != mask->k_tokens) return PVA_ERR_INVALID_ARG;
    const int64_t n = ((int64_t)mask->q_tokens + chunk_size - 1) / chunk_size;
    if (n == 0) return PVA_OK;
    if (n > INT32_MAX) return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    chunk_area_kernel<<<(unsigned)n, kAreaThreads, 0, st>>>(
        cu_seqlens_dev, num_docs, mask->kind, mask->window, mask->num_prefix_docs,
        mask->q_tokens, chunk_size, areas_dev);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" pva_status pva_dispatch_chunks(const int64_t* areas_dev, int32_t num_chunks,
                                          int32_t cp, int32_t* bucket_dev,
                                          int64_t* bucket_area_dev, void* stream) {
    if (!areas_dev || !bucket_dev || !bucket_area_dev || cp <= 0 || num_chunks < 0 ||
        num_chunks % cp != 0)
        return PVA_ERR_INVALID_ARG;
    if (num_chunks > kMaxDispatchChunks || cp > kMaxDispatchBuckets) return PVA_ERR_UNSUPPORTED;
    if (num_chunks == 0) return PVA_OK;
    const size_t smem = dispatch_smem(num_chunks, cp);
    if (cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return PVA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    dispatch_kernel<<<1, kDispatchThreads, smem, st>>>(areas_dev, num_chunks, cp, bucket_dev,
                                                       bucket_area_dev);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" int32_t pva_striped_shard_len(int32_t total_tokens, int32_t cp, int32_t rank,
                                         int32_t stripe) {
    if (total_tokens < 0 || cp <= 0 || rank < 0 || rank >= cp || stripe <= 0) return -1;
    int64_t n = 0;
    for (int64_t s = rank; s * stripe < total_tokens; s += cp) {
        const int64_t e = (s + 1) * stripe < total_tokens ? (s + 1) * stripe : total_tokens;
        n += e - s * stripe;
    }
    return (int32_t)n;
}

extern "C" pva_status pva_striped_shard(int32_t total_tokens, int32_t cp, int32_t rank,
                                        int32_t stripe, int32_t* map_dev, void* stream) {
    const int32_t n = pva_striped_shard_len(total_tokens, cp, rank, stripe);
    if (n < 0 || !map_dev) return PVA_ERR_INVALID_ARG;
    if (n == 0) return PVA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int threads = 256;
    int blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    striped_kernel<<<blocks, threads, 0, st>>>(total_tokens, cp, rank, stripe, n, map_dev);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" int32_t pva_wlb_choose(const int32_t* cu_seqlens_host, int32_t num_docs, int32_t cp,
                                  int32_t tile, int32_t head_dim, int64_t* costs_host) {
    if (!cu_seqlens_host || !costs_host || num_docs < 0 || cp <= 0 || tile <= 0 ||
        head_dim <= 0)
        return -1;
    const int32_t* cu = cu_seqlens_host;
    if (cu[0] != 0) return -1;
    for (int32_t d = 0; d < num_docs; ++d)
        if (cu[d + 1] < cu[d]) return -1;
    const int32_t T = cu[num_docs];
    std::vector<int64_t> seq(cp, 0), doc(cp, 0);
    for (int32_t r = 0; r < cp; ++r) {
        const int32_t chunks[2] = {r, 2 * cp - 1 - r};
        for (int e = 0; e < 2; ++e) {
            int32_t off, len;
            zz_chunk(T, cp, chunks[e], &off, &len);
            // documents that meet [off, off + len): binary search for the first
            int32_t lo = 0, hi = num_docs;
            while (lo < hi) {
                const int32_t mid = (lo + hi) >> 1;
                if (cu[mid + 1] <= off) lo = mid + 1;
                else hi = mid;
            }
            for (int32_t d = lo; d < num_docs && cu[d] < off + len; ++d) {
                const int32_t a = off > cu[d] ? off : cu[d];
                const int32_t b = off + len < cu[d + 1] ? off + len : cu[d + 1];
                if (a < b) seq[r] += piece_flops(a - cu[d], b - cu[d], tile, head_dim);
            }
            for (int32_t d = 0; d < num_docs; ++d) {
                zz_chunk(cu[d + 1] - cu[d], cp, chunks[e], &off, &len);
                if (len > 0) doc[r] += piece_flops(off, off + len, tile, head_dim);
            }
        }
    }
    int64_t mseq = 0, mdoc = 0;
    for (int32_t r = 0; r < cp; ++r) {
        costs_host[r] = seq[r];
        costs_host[cp + r] = doc[r];
        if (seq[r] > mseq) mseq = seq[r];
        if (doc[r] > mdoc) mdoc = doc[r];
    }
    return mdoc < mseq ? 1 : 0;
}
