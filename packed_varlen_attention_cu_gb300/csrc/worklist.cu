// worklist.cu -- device construction of the attention worklist.
//
// "03 · 长文负载均衡" §3.2: attention is cut into tiles; Libra TAP charges
// every tile its exact causal query-key pair count and DCP only creates a
// computation block where the mask is not all zero.  §2.1 (VRSP) and
// "数据并行负载均衡" §4.4 (phase 1): LPT -- sort by cost descending and put
// each item on the currently lightest bin.  Here the bins are the persistent
// CTAs of one GPU.
//
// Kernels (all on the caller's stream, no host round trip):
//   wl_plan   1 CTA  : validate cu_seqlens, derive slices and query segments
//                      of the mask, per-segment unit/run bases (block scans)
//   wl_units  grid   : one thread per work unit: kv-tile span of every slice
//                      for its two sub-tiles, exact pair count, cost, sort key
//   wl_sort_chunks / wl_merge_rank : stable sort by (cost desc, uid asc)
//   wl_lpt    1 CTA  : exact LPT in batches (see below), CTA offsets
//   wl_sort_chunks / wl_merge_rank : sort by (cta, uid): each CTA's list in
//                      enumeration order
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/pva.h"
#include "common.h"
#include "wl_layout.cuh"

namespace pva {
namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ void zz_chunk_dev(int32_t len, int32_t cp, int32_t c, int32_t& off,
                                             int32_t& clen) {
    const int32_t n = 2 * cp, base = len / n, rem = len % n;
    clen = base + (c < rem ? 1 : 0);
    off = c * base + (c < rem ? c : rem);
}

// Block-wide exclusive scan of N int32 lanes per thread (blockDim = 1024).
template <int N>
__device__ void block_scan_excl(int32_t (&v)[N], int32_t (&tot)[N], int32_t (*sm)[N]) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t inc[N];
#pragma unroll
    for (int k = 0; k < N; ++k) inc[k] = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            int32_t t = __shfl_up_sync(0xffffffffu, inc[k], o);
            if (lane >= o) inc[k] += t;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int k = 0; k < N; ++k) sm[w][k] = inc[k];
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            int32_t x = sm[lane][k];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t t = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += t;
            }
            sm[lane][k] = x;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < N; ++k) {
        int32_t base = w > 0 ? sm[w - 1][k] : 0;
        tot[k] = sm[31][k];
        v[k] = base + inc[k] - v[k];
    }
    __syncthreads();
}

struct PlanArgs {
    WlHeader hinit;  // capacities and offsets computed on the host
    uint8_t* base;
    const int32_t* cu;
    int32_t num_docs, kind, window, num_prefix, cp, q_rank, k_rank, num_slices;
    int32_t tile_m, hq, hkv, q_tokens, k_tokens, ring_step, pack_docs;
};

__device__ __forceinline__ void set_error(WlHeader* h, int32_t code) { atomicCAS(&h->error, 0, code); }

// Slices per document and query segments of the mask (the same rules as the
// header documents for pva_mask_kind).
__global__ void __launch_bounds__(kPlanThreads) wl_plan_kernel(PlanArgs a) {
    WlHeader* h = reinterpret_cast<WlHeader*>(a.base);
    WlSlice* slices = reinterpret_cast<WlSlice*>(a.base + a.hinit.off.slices);
    WlSeg* segs = reinterpret_cast<WlSeg*>(a.base + a.hinit.off.segs);
    int32_t* scan = reinterpret_cast<int32_t*>(a.base + a.hinit.off.doc_scan);
    uint32_t* smask = reinterpret_cast<uint32_t*>(a.base + a.hinit.off.smask);
    const int tid = threadIdx.x;
    const int nd = a.num_docs;
    __shared__ int32_t sm4[32][4];
    __shared__ int32_t carry[4];
    __shared__ int32_t s_bad, s_npref, s_nseg, s_nsl;

    if (tid == 0) {
        s_bad = 0;
        s_npref = 0;
        *h = a.hinit;  // error word, counts and sums start at zero
        for (int k = 0; k < 4; ++k) carry[k] = 0;
    }
    if (tid < 64)
        reinterpret_cast<unsigned long long*>(a.base + a.hinit.off.cls_work)[tid] = 0ULL;
    __syncthreads();

    if (a.kind != PVA_MASK_SLICES) {
        if (tid == 0 && a.cu[0] != 0) s_bad = 1;
        for (int d = tid; d < nd; d += kPlanThreads) {
            const int32_t len = a.cu[d + 1] - a.cu[d];
            if (len < 0) s_bad = 1;
            if (a.kind == PVA_MASK_SHARED_QUESTION && d < a.num_prefix && len > 0)
                atomicAdd(&s_npref, 1);
        }
        __syncthreads();
        const int32_t total = a.cu[nd];
        if (a.kind != PVA_MASK_ZIGZAG_PAIR && (total != a.q_tokens || total != a.k_tokens))
            s_bad = 1;
        __syncthreads();
        if (s_bad) {
            if (tid == 0) set_error(h, kErrBadWorklist);
            return;
        }
        // Items: the documents, or for a zigzag ring step the (rank, document)
        // pairs in rank-major order (the order of the ring-ordered Q / K rows).
        const bool ring = a.kind == PVA_MASK_ZIGZAG_STEP;
        const int32_t items = ring ? a.cp * nd : nd;
        // zigzag pair / ring step: the query rank and the key rank of item i
        auto ranks_of = [&](int i, int32_t& qr, int32_t& kr) {
            qr = ring ? i / nd : a.q_rank;
            kr = ring ? (qr - a.ring_step + a.cp) % a.cp : a.k_rank;
        };
        // Short documents sharing tiles (per-document masks, pack_docs): a run of
        // consecutive documents shorter than a tile is cut greedily, in order,
        // into groups of at most tile_m rows; a group holding two or more
        // non-empty documents becomes one query segment with one packed slice.
        // grp[d]: first document of d's packed group (-1: d is not packed);
        // gend[head]: one past the group's last document.
        int32_t* grp = scan + 4 * (items + 1);
        int32_t* gend = scan + 5 * (items + 1);
        const bool pack = a.pack_docs != 0 &&
                          (a.kind == PVA_MASK_CAUSAL || a.kind == PVA_MASK_SLIDING_WINDOW);
        if (pack) {
            auto short_doc = [&](int32_t d) { return a.cu[d + 1] - a.cu[d] < a.tile_m; };
            for (int d = tid; d < nd; d += kPlanThreads) {
                if (!short_doc(d)) {
                    grp[d] = -1;
                    continue;
                }
                if (d > 0 && short_doc(d - 1)) continue;  // not the first of its run
                // this thread cuts the whole run of short documents starting at d
                int32_t x = d;
                while (x < nd && short_doc(x)) {
                    const int32_t head = x;
                    int32_t rows = a.cu[x + 1] - a.cu[x], nonempty = rows > 0, y = x + 1;
                    while (y < nd && short_doc(y) && rows + (a.cu[y + 1] - a.cu[y]) <= a.tile_m) {
                        const int32_t l = a.cu[y + 1] - a.cu[y];
                        rows += l;
                        nonempty += l > 0;
                        ++y;
                    }
                    for (int32_t z = head; z < y; ++z) grp[z] = nonempty >= 2 ? head : -1;
                    if (nonempty >= 2) gend[head] = y;
                    x = y;
                }
            }
            __syncthreads();
        }
        // pass 1: per-item segment / slice counts and zigzag local offsets
        for (int i0 = 0; i0 < items; i0 += kPlanThreads) {
            const int i = i0 + tid;
            int32_t v[4] = {0, 0, 0, 0};
            if (i < items) {
                const int d = ring ? i % nd : i;
                const int32_t len = a.cu[d + 1] - a.cu[d];
                if (a.kind == PVA_MASK_CAUSAL || a.kind == PVA_MASK_SLIDING_WINDOW) {
                    if (pack && grp[d] >= 0) v[0] = v[1] = grp[d] == d;  // the group's head
                    else v[0] = v[1] = len > 0;
                } else if (a.kind == PVA_MASK_SHARED_QUESTION) {
                    v[0] = len > 0;
                    v[1] = len > 0 ? (d >= a.num_prefix ? s_npref + 1 : 1) : 0;
                } else {
                    int32_t qr, kr;
                    ranks_of(i, qr, kr);
                    const int32_t qc[2] = {qr, 2 * a.cp - 1 - qr};
                    const int32_t kc[2] = {kr, 2 * a.cp - 1 - kr};
                    int32_t qo[2], ql[2], ko[2], kl[2];
                    for (int e = 0; e < 2; ++e) {
                        zz_chunk_dev(len, a.cp, qc[e], qo[e], ql[e]);
                        zz_chunk_dev(len, a.cp, kc[e], ko[e], kl[e]);
                    }
                    for (int e = 0; e < 2; ++e) {
                        if (ql[e] <= 0) continue;
                        v[0] += 1;
                        for (int f = 0; f < 2; ++f)
                            if (kl[f] > 0 && ko[f] <= qo[e] + ql[e] - 1) v[1] += 1;
                    }
                    v[2] = ql[0] + ql[1];
                    v[3] = kl[0] + kl[1];
                }
            }
            int32_t tot[4];
            block_scan_excl<4>(v, tot, sm4);
            if (i < items) {
                for (int k = 0; k < 4; ++k) scan[k * (items + 1) + i] = carry[k] + v[k];
            }
            __syncthreads();
            if (tid == 0)
                for (int k = 0; k < 4; ++k) carry[k] += tot[k];
            __syncthreads();
        }
        if (tid == 0) {
            for (int k = 0; k < 4; ++k) scan[k * (items + 1) + items] = carry[k];
            s_nseg = carry[0];
            s_nsl = carry[1];
            if ((a.kind == PVA_MASK_ZIGZAG_PAIR || ring) &&
                (carry[2] != a.q_tokens || carry[3] != a.k_tokens))
                s_bad = 1;
            if (carry[0] > h->cap_segs || carry[1] > h->cap_slices) s_bad = 2;
        }
        __syncthreads();
        if (s_bad) {
            if (tid == 0) set_error(h, s_bad == 2 ? kErrCapacity : kErrBadWorklist);
            return;
        }
        // pass 2: write the slices and segments of every item
        for (int i = tid; i < items; i += kPlanThreads) {
            const int d = ring ? i % nd : i;
            const int32_t len = a.cu[d + 1] - a.cu[d];
            int32_t sg = scan[i], sl = scan[(items + 1) + i];
            if (a.kind == PVA_MASK_CAUSAL || a.kind == PVA_MASK_SLIDING_WINDOW) {
                const int32_t w = a.kind == PVA_MASK_SLIDING_WINDOW ? a.window : 0;
                if (pack && grp[d] >= 0) {
                    if (grp[d] != d) continue;
                    // the group [d, gend[d]): its rows, and the rows that start a document
                    const int32_t g0 = a.cu[d], rows = a.cu[gend[d]] - g0;
                    uint32_t m[4] = {0u, 0u, 0u, 0u};
                    for (int32_t z = d; z < gend[d]; ++z)
                        if (a.cu[z + 1] > a.cu[z]) {
                            const int32_t r = a.cu[z] - g0;
                            m[r >> 5] |= 1u << (r & 31);
                        }
                    slices[sl] = WlSlice{g0, rows, 0, g0, rows, 0, kSlicePacked, w};
                    reinterpret_cast<uint4*>(smask)[sl] = make_uint4(m[0], m[1], m[2], m[3]);
                    segs[sg] = WlSeg{g0, rows, 0, sl, 1, 0, 0, 0};
                    continue;
                }
                if (len <= 0) continue;
                slices[sl] = WlSlice{a.cu[d], len, 0, a.cu[d], len, 0, PVA_SLICE_CAUSAL, w};
                segs[sg] = WlSeg{a.cu[d], len, 0, sl, 1, 0, 0, 0};
            } else if (a.kind == PVA_MASK_SHARED_QUESTION) {
                if (len <= 0) continue;
                const int32_t first = sl;
                if (d >= a.num_prefix) {
                    for (int q = 0; q < a.num_prefix; ++q) {
                        const int32_t ql = a.cu[q + 1] - a.cu[q];
                        if (ql <= 0) continue;
                        slices[sl++] = WlSlice{a.cu[d], len, 0, a.cu[q], ql, 0, PVA_SLICE_FULL, 0};
                    }
                }
                slices[sl++] = WlSlice{a.cu[d], len, 0, a.cu[d], len, 0, PVA_SLICE_CAUSAL, 0};
                segs[sg] = WlSeg{a.cu[d], len, 0, first, sl - first, 0, 0, 0};
            } else {
                int32_t qr, kr;
                ranks_of(i, qr, kr);
                const int32_t qc[2] = {qr, 2 * a.cp - 1 - qr};
                const int32_t kc[2] = {kr, 2 * a.cp - 1 - kr};
                int32_t qo[2], ql[2], ko[2], kl[2];
                for (int e = 0; e < 2; ++e) {
                    zz_chunk_dev(len, a.cp, qc[e], qo[e], ql[e]);
                    zz_chunk_dev(len, a.cp, kc[e], ko[e], kl[e]);
                }
                // first Q row of the item; its K rows: in a pair's K shard, the
                // item's own k-length scan; in ring order, where rank kr's rows
                // of document d start (the query-row scan of item (kr, d))
                const int32_t qloc = scan[2 * (items + 1) + i];
                const int32_t kloc =
                    ring ? scan[2 * (items + 1) + kr * nd + d] : scan[3 * (items + 1) + i];
                const int32_t krow[2] = {kloc, kloc + kl[0]};
                int32_t qrow = qloc;
                for (int e = 0; e < 2; ++e) {
                    if (ql[e] > 0) {
                        const int32_t first = sl;
                        for (int f = 0; f < 2; ++f) {
                            if (kl[f] <= 0 || ko[f] > qo[e] + ql[e] - 1) continue;
                            slices[sl++] =
                                WlSlice{qrow, ql[e], qo[e], krow[f], kl[f], ko[f], PVA_SLICE_CAUSAL, 0};
                        }
                        segs[sg++] = WlSeg{qrow, ql[e], qo[e], first, sl - first, 0, 0, 0};
                    }
                    qrow += ql[e];
                }
            }
        }
    } else {
        // explicit slices (copied by the host): group consecutive equal q ranges
        const int32_t ns = a.num_slices;
        for (int i0 = 0; i0 < ns; i0 += kPlanThreads) {
            const int i = i0 + tid;
            int32_t v[1] = {0};
            if (i < ns) {
                const WlSlice s = slices[i];
                if (i == 0) {
                    v[0] = 1;
                } else {
                    const WlSlice p = slices[i - 1];
                    v[0] = (p.q_row0 != s.q_row0 || p.q_len != s.q_len || p.q_pos0 != s.q_pos0);
                }
            }
            const int32_t flag = v[0];
            int32_t tot[1];
            int32_t(*sm1)[1] = reinterpret_cast<int32_t(*)[1]>(&sm4[0][0]);
            block_scan_excl<1>(v, tot, sm1);
            if (i < ns && flag) {
                const WlSlice s = slices[i];
                const int32_t g = carry[0] + v[0];
                if (g < h->cap_segs) segs[g] = WlSeg{s.q_row0, s.q_len, s.q_pos0, i, 0, 0, 0, 0};
            }
            __syncthreads();
            if (tid == 0) carry[0] += tot[0];
            __syncthreads();
        }
        if (tid == 0) {
            s_nseg = carry[0];
            s_nsl = ns;
            if (carry[0] > h->cap_segs || ns > h->cap_slices) s_bad = 2;
        }
        __syncthreads();
        if (s_bad) {
            if (tid == 0) set_error(h, kErrCapacity);
            return;
        }
        for (int g = tid; g < s_nseg; g += kPlanThreads) {
            const int32_t next = (g + 1 < s_nseg) ? segs[g + 1].slice_begin : ns;
            segs[g].slice_count = next - segs[g].slice_begin;
        }
    }
    __syncthreads();

    // per segment: q tiles, units and runs, then their exclusive scans
    const int32_t nseg = s_nseg;
    const int32_t G = a.hq / a.hkv;
    if (tid == 0)
        for (int k = 0; k < 4; ++k) carry[k] = 0;
    __syncthreads();
    for (int g0 = 0; g0 < nseg; g0 += kPlanThreads) {
        const int g = g0 + tid;
        int32_t v[2] = {0, 0};
        int32_t nt = 0;
        if (g < nseg) {
            const WlSeg s = segs[g];
            nt = (s.q_len + a.tile_m - 1) / a.tile_m;
            const int32_t u = a.hkv * ((G / 2) * nt + (G % 2) * ((nt + 1) / 2));
            v[0] = u;
            v[1] = u * s.slice_count;
        }
        int32_t tot[2];
        int32_t(*sm2)[2] = reinterpret_cast<int32_t(*)[2]>(&sm4[0][0]);
        block_scan_excl<2>(v, tot, sm2);
        if (g < nseg) {
            segs[g].unit_base = carry[0] + v[0];
            segs[g].run_base = carry[1] + v[1];
            segs[g].ntiles = nt;
        }
        __syncthreads();
        if (tid == 0) {
            carry[0] += tot[0];
            carry[1] += tot[1];
        }
        __syncthreads();
    }
    if (tid == 0) {
        h->nsegs = nseg;
        h->nslices = s_nsl;
        if (carry[0] > h->cap_units || carry[1] > h->cap_runs) {
            set_error(h, kErrCapacity);
        } else {
            h->nunits = carry[0];
            h->nruns = carry[1];
        }
    }
}

// kv-tile span [lo_t, hi_t) and allowed-pair count of q tile t against slice
// s, by the whole warp: lane l takes rows r0 + l, r0 + l + 32, ...
__device__ void tile_span_warp(const WlSeg& g, const WlSlice& s, const uint32_t* pm, int32_t t,
                               int32_t tile_m, int32_t tile_n, int32_t& lo_t, int32_t& hi_t,
                               long long& pairs) {
    long long mn = 0x7fffffffffffffffLL, mx = -1, cnt = 0;
    const int32_t r0 = t * tile_m;
    const int32_t r1 = min(r0 + tile_m, g.q_len);
    for (int32_t r = r0 + (int32_t)(threadIdx.x & 31); r < r1; r += 32) {
        int64_t lo, hi;
        slice_keys_of_query(s, (int64_t)s.q_pos0 + r, lo, hi, pm);
        if (hi <= lo) continue;
        cnt += hi - lo;
        mn = lo < mn ? lo : mn;
        mx = hi > mx ? hi : mx;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        const long long a = __shfl_xor_sync(0xffffffffu, mn, o);
        const long long b = __shfl_xor_sync(0xffffffffu, mx, o);
        mn = a < mn ? a : mn;
        mx = b > mx ? b : mx;
    }
    if (cnt == 0) {
        lo_t = hi_t = 0;
    } else {
        // slice-local key indices: 0 <= mn < mx <= k_len < 2^31
        lo_t = (int32_t)mn / tile_n;
        hi_t = (int32_t)(((uint32_t)mx + (uint32_t)tile_n - 1u) / (uint32_t)tile_n);
    }
    pairs = cnt;
}

struct UnitArgs {
    uint8_t* base;
    int32_t tile_m, tile_n, hq, hkv;
    long long c_tile;
};

constexpr int kUnitWarps = 8;  // units per block of the units kernel

// One warp per unit (every lane computes the same unit; the row loops are
// split across lanes).  Enumeration inside a segment: kv head, then head
// pairs (2p, 2p+1) x q tiles, then the odd last head's q-tile pairs.
__global__ void __launch_bounds__(kUnitWarps * 32) wl_units_kernel(UnitArgs a) {
    WlHeader* h = reinterpret_cast<WlHeader*>(a.base);
    if (h->error) return;
    const int32_t n = h->nunits;
    if ((int64_t)blockIdx.x * kUnitWarps >= n) return;
    __shared__ unsigned long long bsum[kUnitWarps][2];
    __shared__ long long bcost[kUnitWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t u = blockIdx.x * kUnitWarps + warp;
    unsigned long long pairs_out = 0, tiles_out = 0;
    long long cost_out = -1;  // -1: no unit
    if (u < n) {
        const WlSlice* slices = reinterpret_cast<const WlSlice*>(a.base + h->off.slices);
        const WlSeg* segs = reinterpret_cast<const WlSeg*>(a.base + h->off.segs);
        WlUnit* units = reinterpret_cast<WlUnit*>(a.base + h->off.units_enum);
        unsigned long long* keys = reinterpret_cast<unsigned long long*>(a.base + h->off.keys);
        WlRun* runs = reinterpret_cast<WlRun*>(a.base + h->off.runs);
        // segment: last g with unit_base <= u
        int32_t lo = 0, hi = h->nsegs - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (segs[mid].unit_base <= u) lo = mid;
            else hi = mid - 1;
        }
        const int32_t gi = lo;
        const WlSeg g = segs[gi];
        const int32_t G = a.hq / a.hkv, nt = g.ntiles;
        const int32_t per_kvh = (G / 2) * nt + (G % 2) * ((nt + 1) / 2);
        const int32_t e = u - g.unit_base;
        WlUnit w;
        w.uid = u;
        w.seg = gi;
        w.kvh = e / per_kvh;
        const int32_t e2 = e % per_kvh;
        if (e2 < (G / 2) * nt) {
            const int32_t p = e2 / nt, t = e2 % nt;
            w.t0 = w.t1 = t;
            w.h0 = w.kvh * G + 2 * p;
            w.h1 = w.h0 + 1;
        } else {
            const int32_t uu = e2 - (G / 2) * nt;
            w.t0 = 2 * uu;
            w.t1 = (2 * uu + 1 < nt) ? 2 * uu + 1 : -1;
            w.h0 = w.kvh * G + G - 1;
            w.h1 = w.t1 >= 0 ? w.h0 : -1;
        }
        const int nsub = w.h1 >= 0 ? 2 : 1;
        w.run_begin = g.run_base + e * g.slice_count;
        w.run_count = g.slice_count;
        w.cta = -1;
        w.pad = 0;
        long long pairs = 0, tiles = 0;
        int32_t ntiles = 0;
        for (int32_t si = 0; si < g.slice_count; ++si) {
            const WlSlice sl = slices[g.slice_begin + si];
            const uint32_t* pm = slice_mask(a.base, h, sl, g.slice_begin + si);
            int32_t rlo = 0, rhi = 0;
            bool have = false;
            const int32_t ts[2] = {w.t0, w.t1};
            for (int k = 0; k < nsub; ++k) {
                int32_t a0, b0;
                long long pr;
                tile_span_warp(g, sl, pm, ts[k], a.tile_m, a.tile_n, a0, b0, pr);
                pairs += pr;
                if (b0 > a0) {
                    if (!have || a0 < rlo) rlo = a0;
                    if (!have || b0 > rhi) rhi = b0;
                    have = true;
                }
            }
            if (lane == 0) runs[w.run_begin + si] = WlRun{g.slice_begin + si, rlo, rhi, 0};
            tiles += (long long)(rhi - rlo) * nsub;
            ntiles += rhi - rlo;
        }
        w.ntiles = ntiles;
        w.pairs = pairs;
        w.cost = pairs + a.c_tile * (tiles + nsub);
        if (lane == 0) {
            units[u] = w;
            if (w.cost < 0 || w.cost >= (1LL << kCostBits)) set_error(h, kErrCostRange);
            const unsigned long long inv = ((1ULL << kCostBits) - 1) - (unsigned long long)w.cost;
            keys[u] = (inv << kUidBits) | (unsigned long long)u;
        }
        pairs_out = (unsigned long long)pairs;
        tiles_out = (unsigned long long)tiles;
        cost_out = w.cost;
    }
    if (lane == 0) {
        bsum[warp][0] = pairs_out;
        bsum[warp][1] = tiles_out;
        bcost[warp] = cost_out;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long p = 0, q = 0;
        for (int i = 0; i < kUnitWarps; ++i) {
            p += bsum[i][0];
            q += bsum[i][1];
        }
        atomicAdd(&h->pair_sum, p);
        atomicAdd(&h->tile_sum, q);
        if (h->dispatch == PVA_DISPATCH_DYNAMIC) {
            // summed cost per dispatch class: one atomic per class in the block
            unsigned long long* cw =
                reinterpret_cast<unsigned long long*>(a.base + h->off.cls_work);
            for (int i = 0; i < kUnitWarps; ++i) {
                if (bcost[i] < 0) continue;
                const int32_t ci = dispatch_class(bcost[i]);
                bool seen = false;
                for (int j = 0; j < i; ++j) seen |= bcost[j] >= 0 && dispatch_class(bcost[j]) == ci;
                if (seen) continue;
                unsigned long long sum = 0;
                for (int j = i; j < kUnitWarps; ++j)
                    if (bcost[j] >= 0 && dispatch_class(bcost[j]) == ci) sum += bcost[j];
                atomicAdd(&cw[ci], sum);
            }
        }
    }
}

// Stable sort by (cost desc, uid asc).  Every key is unique, so a unit's
// rank is the number of smaller keys.  Two kernels: each 2048-key chunk is
// sorted in shared memory (bitonic network), then every key's rank is its
// position in its own chunk plus its lower bound in each other chunk.
constexpr int kSortChunk = 2048;
constexpr int kSortThreads = 1024;

// What the sort kernels work on: n keys (a device count, read when the kernel
// runs), and where a failed earlier stage left its error word.
struct SortArgs {
    const int32_t* err;
    const int32_t* n;
    const unsigned long long* cls_work;  // summed cost per class (dispatch keys only)
    int32_t* split;                      // where block 0 records the split class
    int32_t num_ctas;                    // CTAs of the forward launch
    unsigned long long* keys;
    int32_t* order;             // rank -> uid (LPT order)
    int32_t* dorder;            // rank -> uid (dispatch order)
    const WlUnit* units_enum;   // CTA order: units by uid ...
    WlUnit* units;              // ... written at their rank
};

// kDispatchKeys: the chunk's keys are made here from the units (class desc,
// uid asc) instead of read from `keys`.
template <bool kDispatchKeys>
__global__ void __launch_bounds__(kSortThreads) wl_sort_chunks_kernel(SortArgs a) {
    if (*a.err) return;
    const int32_t n = *a.n;
    const int32_t c0 = blockIdx.x * kSortChunk;
    if (c0 >= n) return;
    unsigned long long* keys = a.keys;
    __shared__ unsigned long long sk[kSortChunk];
    __shared__ int32_t s_split;
    const int32_t m = min(kSortChunk, n - c0);
    if (kDispatchKeys) {
        // the split: the highest non-empty class c with less work below it than
        // num_ctas * 2^(c+1) (capped at 38)
        // one warp: lane l holds classes l and l + 32; an exclusive prefix sum over
        // the 64 class totals gives each class the work below it (one thread walking
        // the 64 totals spent ~20 us in dependent L2 loads)
        if (threadIdx.x < 32) {
            const unsigned full = 0xffffffffu;
            const int lane = threadIdx.x;
            const unsigned long long w0 = a.cls_work[lane], w1 = a.cls_work[lane + 32];
            unsigned long long p0 = w0, p1 = w1;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long x0 = __shfl_up_sync(full, p0, o);
                const unsigned long long x1 = __shfl_up_sync(full, p1, o);
                if (lane >= o) {
                    p0 += x0;
                    p1 += x1;
                }
            }
            p1 += __shfl_sync(full, p0, 31);  // classes 32.. also sit above all of 0..31
            const unsigned long long B = (unsigned long long)a.num_ctas;
            // class c qualifies: non-empty, and less work under it than B * 2^(c+1)
            const int s0 = lane + 1, s1 = lane + 33 < 63 ? lane + 33 : 63;
            const bool q0 = w0 != 0 && p0 - w0 < (B << s0);
            const bool q1 = w1 != 0 && p1 - w1 < (B << s1);
            const unsigned m0 = __ballot_sync(full, q0), m1 = __ballot_sync(full, q1);
            // the highest qualifying class, capped at 38 (0 when none qualifies)
            int32_t split = m1 ? 63 - __clz(m1) : (m0 ? 31 - __clz(m0) : 0);
            split = split < 38 ? split : 38;
            if (lane == 0) {
                s_split = split;
                if (blockIdx.x == 0) *a.split = split;
            }
        }
        __syncthreads();
    }
    // Bitonic sort of the smallest power of two >= max(m, 64) keys (the tail of a
    // chunk is padding, ~0).  Warp w holds keys [64 w, 64 w + 64) in registers, two
    // per lane (k0 = key 64 w + 2 lane, k1 the next): every stage with a stride of
    // at most 32 runs there with shuffles, only the wider ones go through shared
    // memory.  Same network and result as the all-shared-memory form.
    int32_t np2 = 64;
    while (np2 < m) np2 <<= 1;
    const int32_t e0 = 2 * (int32_t)threadIdx.x;  // index of k0
    const bool holds = e0 < np2;
    auto key_at = [&](int32_t i) -> unsigned long long {
        unsigned long long key = ~0ULL;
        if (i < m) {
            if (kDispatchKeys) {
                // above the split: (0, 63 - class, uid); else (1, 2^39 - 1 - cost, uid)
                const long long c = a.units_enum[c0 + i].cost;
                const int32_t cls = dispatch_class(c);
                key = cls > s_split
                          ? ((unsigned long long)(63 - cls) << 57)
                          : (1ULL << 63) | ((((1ULL << 39) - 1) - (unsigned long long)c) << kUidBits);
                key |= (unsigned long long)(c0 + i);
            } else {
                key = keys[c0 + i];
            }
        }
        return key;
    };
    unsigned long long k0 = holds ? key_at(e0) : ~0ULL, k1 = holds ? key_at(e0 + 1) : ~0ULL;
    // stages stride = top .. 1 of merge size `size` on the warp's registers; the pair
    // (lo, lo + stride) ends ascending when (lo & size) == 0, descending otherwise
    auto warp_stages = [&](int32_t size, int32_t top) {
        for (int32_t stride = top; stride > 0; stride >>= 1) {
            if (stride == 1) {
                const bool up = (e0 & size) == 0;
                if ((k0 > k1) == up) {
                    const unsigned long long t = k0;
                    k0 = k1;
                    k1 = t;
                }
            } else {
                const unsigned long long o0 = __shfl_xor_sync(0xffffffffu, k0, stride >> 1);
                const unsigned long long o1 = __shfl_xor_sync(0xffffffffu, k1, stride >> 1);
                const bool lower = (e0 & stride) == 0;
                const bool up = ((lower ? e0 : e0 - stride) & size) == 0;
                const bool keep_min = lower == up;
                k0 = keep_min ? (k0 < o0 ? k0 : o0) : (k0 > o0 ? k0 : o0);
                k1 = keep_min ? (k1 < o1 ? k1 : o1) : (k1 > o1 ? k1 : o1);
            }
        }
    };
    for (int32_t size = 2; size <= 64; size <<= 1) warp_stages(size, size >> 1);
    for (int32_t size = 128; size <= np2; size <<= 1) {
        if (holds) {
            sk[e0] = k0;
            sk[e0 + 1] = k1;
        }
        __syncthreads();
        for (int32_t stride = size >> 1; stride >= 64; stride >>= 1) {
            for (int32_t t = threadIdx.x; t < np2 / 2; t += kSortThreads) {
                const int32_t lo = 2 * t - (t & (stride - 1));
                const int32_t hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long x = sk[lo], y = sk[hi];
                if ((x > y) == up) {
                    sk[lo] = y;
                    sk[hi] = x;
                }
            }
            __syncthreads();
        }
        if (holds) {
            k0 = sk[e0];
            k1 = sk[e0 + 1];
        }
        warp_stages(size, 32);
        __syncthreads();  // every warp has read its keys before the next size rewrites them
    }
    static_assert(kSortChunk / 2 == kSortThreads, "two keys per thread");
    if (e0 < m) keys[c0 + e0] = k0;
    if (e0 + 1 < m) keys[c0 + e0 + 1] = k1;
}

// kMode kRankLpt: keys are (~cost, uid) and order[rank] = uid (LPT order).
// kRankCta: keys are (cta, uid) and units[rank] = the unit with its CTA, i.e.
// the CSR list of every CTA in enumeration order.
// kRankDispatch: keys are (63 - class, uid) and dorder[rank] = uid.
enum RankMode { kRankLpt = 0, kRankCta = 1, kRankDispatch = 2 };
template <int kMode>
__global__ void __launch_bounds__(kSortThreads) wl_merge_rank_kernel(SortArgs a) {
    if (*a.err) return;
    const int32_t n = *a.n;
    const int32_t c0 = blockIdx.x * kSortChunk;
    if (c0 >= n) return;
    const unsigned long long* keys = a.keys;
    __shared__ unsigned long long other[kSortChunk];
    const int32_t m = min(kSortChunk, n - c0);
    const int32_t nchunks = (n + kSortChunk - 1) / kSortChunk;
    unsigned long long mine[2];
    int32_t rank[2];
    for (int e = 0; e < 2; ++e) {
        const int32_t i = threadIdx.x + e * kSortThreads;
        mine[e] = i < m ? keys[c0 + i] : ~0ULL;
        rank[e] = i;
    }
    for (int32_t c = 0; c < nchunks; ++c) {
        if (c == (int32_t)blockIdx.x) continue;
        const int32_t oc = c * kSortChunk, om = min(kSortChunk, n - oc);
        __syncthreads();
        for (int32_t i = threadIdx.x; i < om; i += kSortThreads) other[i] = keys[oc + i];
        __syncthreads();
        for (int e = 0; e < 2; ++e) {
            int32_t lo = 0, hi = om;  // number of keys < mine[e]
            while (lo < hi) {
                const int32_t mid = (lo + hi) >> 1;
                if (other[mid] < mine[e]) lo = mid + 1;
                else hi = mid;
            }
            rank[e] += lo;
        }
    }
    for (int e = 0; e < 2; ++e) {
        const int32_t i = threadIdx.x + e * kSortThreads;
        if (i >= m) continue;
        const int32_t uid = (int32_t)(mine[e] & ((1ULL << kUidBits) - 1));
        if (kMode == kRankCta) {
            WlUnit x = a.units_enum[uid];
            x.cta = (int32_t)(mine[e] >> kUidBits);
            a.units[rank[e]] = x;
        } else if (kMode == kRankDispatch) {
            a.dorder[rank[e]] = uid;
        } else {
            a.order[rank[e]] = uid;
        }
    }
}

// LPT over num_ctas bins, exact and in parallel batches.
// Bins are kept sorted by (load, id) as composite keys (load << 10 | id).
// With tasks t, t+1, ... in LPT order, sequential LPT sends task t+j to the
// j-th lightest bin S_j as long as S_j is lighter than every bin that
// received a task earlier in the batch, i.e. S_j < min_{i<j} (S_i + c_{t+i});
// the first j where this fails ends the batch.  If it fails at j = 1, task
// t+1 goes to S_0 again: a run of consecutive tasks then goes to S_0 while
// S_0 plus their cost prefix stays below S_1.  After each step the bins are
// re-sorted by rank counting, split F ways across the block.
constexpr int kLptStage = 1024;

__device__ __forceinline__ void lpt_resort(unsigned long long* S, const unsigned long long* Snew,
                                           int32_t* rc, int32_t B, int32_t Bp, int32_t F) {
    const int tid = threadIdx.x;
    const int32_t j = tid % Bp, q = tid / Bp;
    const int32_t chunk = (B + F - 1) / F;
    if (j < B && q < F) {
        const unsigned long long me = Snew[j];
        const int32_t i1 = min(B, (q + 1) * chunk);
        int32_t r = 0;
#pragma unroll 4
        for (int32_t i = q * chunk; i < i1; ++i) r += Snew[i] < me;
        rc[q * Bp + j] = r;
    }
    __syncthreads();
    if (tid < B) {
        int32_t r = 0;
        for (int32_t qq = 0; qq < F; ++qq) r += rc[qq * Bp + tid];
        S[r] = Snew[tid];
    }
    __syncthreads();
}

// Move/swap refinement after LPT ("数据并行负载均衡" §4.4, phase 2), by the
// whole block: each round takes the most and the least loaded bins (ties:
// lower id) and stops once their gap is under 5% of the larger load.  The
// heavy bin's costliest unit x and the light bin's cheapest unit y (ties:
// lower uid) are found by block-wide scans; moving x or swapping x and y,
// whichever leaves the smaller gap between the two bins (a move on a tie), is
// applied if it shrinks the gap, else the refinement ends.
__device__ void lpt_refine(WlHeader* h, const WlUnit* units_enum, int32_t* assign,
                           const unsigned long long* S, int32_t* cnt, int32_t n, int32_t B) {
    __shared__ long long load[kMaxBins];
    __shared__ unsigned long long rx[32], ry[32];
    __shared__ int32_t r_bmax, r_bmin, r_go;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = (blockDim.x + 31) >> 5;
    for (int32_t i = tid; i < B; i += blockDim.x) load[S[i] & 1023ULL] = (long long)(S[i] >> 10);
    __syncthreads();
    int32_t rounds = 0;
    for (int32_t it = 0; it < h->refine_iters; ++it) {
        if (w == 0) {
            long long mx = LLONG_MIN, mn = LLONG_MAX;
            int32_t bx = INT32_MAX, bn = INT32_MAX;
            for (int32_t b = lane; b < B; b += 32) {
                if (load[b] > mx) { mx = load[b]; bx = b; }
                if (load[b] < mn) { mn = load[b]; bn = b; }
            }
            for (int o = 16; o > 0; o >>= 1) {
                const long long omx = __shfl_xor_sync(0xffffffffu, mx, o);
                const int32_t obx = __shfl_xor_sync(0xffffffffu, bx, o);
                const long long omn = __shfl_xor_sync(0xffffffffu, mn, o);
                const int32_t obn = __shfl_xor_sync(0xffffffffu, bn, o);
                if (omx > mx || (omx == mx && obx < bx)) { mx = omx; bx = obx; }
                if (omn < mn || (omn == mn && obn < bn)) { mn = omn; bn = obn; }
            }
            if (lane == 0) {
                r_bmax = bx;
                r_bmin = bn;
                const long long gap = mx - mn;
                r_go = !(gap * 20 < mx || gap == 0);
            }
        }
        __syncthreads();
        if (!r_go) break;
        const int32_t bmax = r_bmax, bmin = r_bmin;
        // x: max of (cost, lowest uid); y: min of (cost, lowest uid)
        unsigned long long kx = 0, ky = ~0ULL;
        for (int32_t u = tid; u < n; u += blockDim.x) {
            const int32_t a = assign[u];
            if (a != bmax && a != bmin) continue;
            const unsigned long long c = (unsigned long long)units_enum[u].cost;
            if (a == bmax) {
                const unsigned long long k = (c << kUidBits) | ((1ULL << kUidBits) - 1 - u);
                if (k > kx) kx = k;  // 0 stays "none": a real key has uid bits < 2^24 - 1 - u
            } else {
                const unsigned long long k = (c << kUidBits) | (unsigned long long)u;
                if (k < ky) ky = k;
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long a = __shfl_xor_sync(0xffffffffu, kx, o);
            const unsigned long long b = __shfl_xor_sync(0xffffffffu, ky, o);
            if (a > kx) kx = a;
            if (b < ky) ky = b;
        }
        if (lane == 0) {
            rx[w] = kx;
            ry[w] = ky;
        }
        __syncthreads();
        if (tid == 0) {
            bool have_x = false;
            unsigned long long bx = 0, by = ~0ULL;
            for (int i = 0; i < nw; ++i) {
                if (rx[i] > bx) bx = rx[i];
                if (ry[i] < by) by = ry[i];
            }
            // a heavy bin always holds a unit (its load is positive); a key of 0
            // would be a unit of cost 0 and uid 2^24 - 1, which the uid bound excludes
            have_x = bx != 0;
            r_go = 0;
            if (have_x) {
                const int32_t x = (int32_t)((1ULL << kUidBits) - 1 - (bx & ((1ULL << kUidBits) - 1)));
                const long long cx = (long long)(bx >> kUidBits);
                const long long gap = load[bmax] - load[bmin];
                long long gm = gap - 2 * cx;
                if (gm < 0) gm = -gm;
                long long gs = LLONG_MAX;
                int32_t y = -1;
                long long cy = 0;
                if (by != ~0ULL) {
                    y = (int32_t)(by & ((1ULL << kUidBits) - 1));
                    cy = (long long)(by >> kUidBits);
                    gs = gap - 2 * (cx - cy);
                    if (gs < 0) gs = -gs;
                }
                if (gm < gap || gs < gap) {
                    if (gm <= gs) {
                        assign[x] = bmin;
                        load[bmax] -= cx;
                        load[bmin] += cx;
                        --cnt[bmax];
                        ++cnt[bmin];
                    } else {
                        assign[x] = bmin;
                        assign[y] = bmax;
                        load[bmax] += cy - cx;
                        load[bmin] += cx - cy;
                    }
                    r_go = 1;
                }
            }
        }
        __syncthreads();
        if (!r_go) break;
        ++rounds;
    }
    if (tid == 0) h->refine_rounds = rounds;
    __syncthreads();
}

__global__ void __launch_bounds__(kMaxBins) wl_lpt_kernel(uint8_t* base, int32_t F) {
    WlHeader* h = reinterpret_cast<WlHeader*>(base);
    if (h->error) return;
    const int32_t n = h->nunits;
    const int32_t B = h->num_ctas;
    const int32_t Bp = (B + 31) & ~31;  // bins rounded up to whole warps
    const WlUnit* units_enum = reinterpret_cast<const WlUnit*>(base + h->off.units_enum);
    const int32_t* order = reinterpret_cast<const int32_t*>(base + h->off.order);
    int32_t* assign = reinterpret_cast<int32_t*>(base + h->off.assign);
    int32_t* cta_off = reinterpret_cast<int32_t*>(base + h->off.cta_off);
    __shared__ unsigned long long S[kMaxBins], Snew[kMaxBins];
    __shared__ int32_t cnt[kMaxBins];
    __shared__ int32_t rc[kMaxBins];
    // the next kLptStage units in LPT order (cost, uid), refilled as t advances
    __shared__ long long scost[kLptStage];
    __shared__ int32_t suid[kLptStage];
    __shared__ unsigned long long wmin[32];
    __shared__ long long wsum[32];
    __shared__ int32_t wint[32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nw = Bp >> 5;           // warps that hold bins
    const bool main = tid < Bp;
    // bin keys hold load << 10: the total cost must stay below 2^53
    const unsigned long long total_cost =
        h->pair_sum + (unsigned long long)h->c_tile * (h->tile_sum + 2ULL * (unsigned)n);
    if (total_cost >= (1ULL << 53)) {
        if (tid == 0) set_error(h, kErrCostRange);
        return;
    }
    if (tid < B) {
        S[tid] = (unsigned long long)tid;
        cnt[tid] = 0;
    }
    __syncthreads();
    int32_t stage0 = -kLptStage, steps = 0;
    for (int32_t t = 0; t < n; ++steps) {
        if (t + Bp > stage0 + kLptStage) {  // a step may read past the staged window
            stage0 = t;
            for (int32_t i = tid; i < kLptStage && t + i < n; i += blockDim.x) {
                const int32_t uid = order[t + i];
                suid[i] = uid;
                scost[i] = units_enum[uid].cost;
            }
            __syncthreads();
        }
        const bool have = tid < B && t + tid < n;
        const long long c = have ? scost[t + tid - stage0] : 0;
        // candidate value of bin j after receiving task t+j; exclusive prefix-min
        const unsigned long long val = have ? S[tid] + ((unsigned long long)c << 10) : ~0ULL;
        unsigned long long inc = val;
        if (main) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long x = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o && x < inc) inc = x;
            }
            if (lane == 31) wmin[w] = inc;
        }
        __syncthreads();
        unsigned long long ex = ~0ULL;
        if (main) {
            ex = __shfl_up_sync(0xffffffffu, inc, 1);
            if (lane == 0) ex = ~0ULL;
            for (int i = 0; i < w; ++i) ex = wmin[i] < ex ? wmin[i] : ex;
            // task t+j goes to S_j iff it exists and S_j < prefix-min (always for j = 0)
            const bool ok = have && (tid == 0 || S[tid] < ex);
            const unsigned fail = __ballot_sync(0xffffffffu, !ok);
            if (lane == 0) wint[w] = fail ? w * 32 + __ffs(fail) - 1 : 0x7fffffff;
        }
        __syncthreads();
        int32_t k = B;
        for (int i = 0; i < nw; ++i) k = min(k, wint[i]);
        __syncthreads();  // wint is reused below
        if (k == 1 && t + 1 < n) {
            // run of consecutive tasks into S_0 (see above)
            const int32_t j = tid;
            const bool in = main && t + j < n && t + j - stage0 < kLptStage;
            const long long cj = in ? scost[t + j - stage0] : 0;
            long long incl = cj;
            if (main) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += x;
                }
                if (lane == 31) wsum[w] = incl;
            }
            __syncthreads();
            const unsigned long long s0 = S[0], s1 = B > 1 ? S[1] : ~0ULL;
            long long excl = incl - cj;
            if (main) {
                for (int i = 0; i < w; ++i) excl += wsum[i];
                const bool go = j >= 1 && in && s0 + ((unsigned long long)excl << 10) < s1;
                const unsigned bal = __ballot_sync(0xffffffffu, go);
                if (lane == 0) wint[w] = __popc(bal);
            }
            __syncthreads();
            int32_t m = 1;
            for (int i = 0; i < nw; ++i) m += wint[i];
            const int32_t bin = (int32_t)(s0 & 1023ULL);
            if (main && j < m) {
                const int32_t uid = suid[t + j - stage0];
                assign[uid] = bin;
            }
            if (main && j == m - 1) Snew[0] = s0 + ((unsigned long long)(excl + cj) << 10);
            if (tid > 0 && tid < B) Snew[tid] = S[tid];
            __syncthreads();
            if (tid == 0) cnt[bin] += m;
            lpt_resort(S, Snew, rc, B, Bp, F);
            t += m;
            continue;
        }
        if (tid < k) {
            const int32_t uid = suid[t + tid - stage0];
            const int32_t bin = (int32_t)(S[tid] & 1023ULL);
            assign[uid] = bin;
            ++cnt[bin];
            Snew[tid] = val;
        } else if (tid < B) {
            Snew[tid] = S[tid];
        }
        __syncthreads();
        lpt_resort(S, Snew, rc, B, Bp, F);
        t += k;
    }
    if (tid == 0) h->lpt_steps = steps;
    if (h->refine_iters > 0 && B > 1) lpt_refine(h, units_enum, assign, S, cnt, n, B);
    // CSR offsets: exclusive scan of the bin counts (warp scans + warp totals)
    int32_t inc = tid < B ? cnt[tid] : 0;
    const int32_t mine = inc;
    if (main) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) wint[w] = inc;
    }
    __syncthreads();
    if (main) {
        int32_t base_w = 0;
        for (int i = 0; i < w; ++i) base_w += wint[i];
        const int32_t excl = base_w + inc - mine;
        if (tid < B) cta_off[tid] = excl;
        if (tid == B - 1) cta_off[B] = excl + mine;
        if (tid < B) rc[tid] = excl;
    }
    __syncthreads();
    // Each CTA runs its units in enumeration order (segment, kv head, head pair,
    // q tile): CTAs that run at the same time then walk the K/V of the same
    // documents, which stay in L2.  Keys (cta, uid) are sorted next.
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(base + h->off.keys);
    for (int32_t u = tid; u < n; u += blockDim.x)
        keys[u] = ((unsigned long long)assign[u] << kUidBits) | (unsigned long long)u;
}

// Backward plan (kv-major units) from the forward worklist's slices, one CTA.
// 1. Sort the slice indices by (k_row0, k_len, index) in shared memory
//    (bitonic); equal key ranges become runs: the key groups.
// 2. A block scan over the groups of their key-tile counts.
// 3. One unit per (group, key tile, kv head) with its cost (q-tile steps over
//    the group's slices and the heads of the kv head's group, + 1) and a sort
//    key.  Static dispatch deals units by cost (desc, uid asc).  Dynamic
//    dispatch claims them by power-of-two cost class (desc); inside a class in
//    uid order, which runs group by group, kv head by kv head, key tiles
//    ascending, so that the CTAs running at the same time read the same
//    documents' query tiles while the classes still put large units first.
constexpr int kBwdPlanThreads = 1024;

__global__ void __launch_bounds__(kBwdPlanThreads)
    bwd_plan_kernel(const uint8_t* wl, uint8_t* plan) {
    extern __shared__ unsigned long long bsm[];
    const WlHeader* h = reinterpret_cast<const WlHeader*>(wl);
    BwdHeader* bh = reinterpret_cast<BwdHeader*>(plan);
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    if (h->error != 0) {
        if (threadIdx.x == 0) bh->error = h->error;
        return;
    }
    const int32_t ns = h->nslices;
    if (ns > kBwdMaxSlices) {
        if (threadIdx.x == 0) bh->error = kErrCapacity;
        return;
    }
    const WlSlice* slices = reinterpret_cast<const WlSlice*>(wl + h->off.slices);
    BwdUnit* units = reinterpret_cast<BwdUnit*>(plan + bh->off_units);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(plan + bh->off_keys);
    int32_t* gsl = reinterpret_cast<int32_t*>(plan + bh->off_gslices);
    const int32_t hkv = bh->hkv, G = bh->hq / bh->hkv;
    const bool dyn = h->dispatch == PVA_DISPATCH_DYNAMIC;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int32_t np2 = 1;
    while (np2 < ns) np2 <<= 1;
    // (k_row0, k_len) packed, k_len < 2^31; the slice index rides in sidx
    unsigned long long* skey = bsm;                               // [np2]
    int32_t* sidx = reinterpret_cast<int32_t*>(bsm + np2);        // [np2]
    int32_t* lead = sidx + np2;                                   // [np2] 1 at a group's first
    for (int32_t i = tid; i < np2; i += kBwdPlanThreads) {
        if (i < ns) {
            const WlSlice sl = slices[i];
            skey[i] = ((unsigned long long)(uint32_t)sl.k_row0 << 32) | (uint32_t)sl.k_len;
        } else {
            skey[i] = ~0ULL;
        }
        sidx[i] = i;
    }
    __syncthreads();
    for (int32_t size = 2; size <= np2; size <<= 1) {
        for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (int32_t t = tid; t < np2 / 2; t += kBwdPlanThreads) {
                const int32_t lo = 2 * t - (t & (stride - 1));
                const int32_t hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long xk = skey[lo], yk = skey[hi];
                const int32_t xi = sidx[lo], yi = sidx[hi];
                const bool x_first = xk < yk || (xk == yk && xi < yi);
                if (x_first != up) {
                    skey[lo] = yk;
                    skey[hi] = xk;
                    sidx[lo] = yi;
                    sidx[hi] = xi;
                }
            }
            __syncthreads();
        }
    }
    for (int32_t i = tid; i < ns; i += kBwdPlanThreads) {
        gsl[i] = sidx[i];
        lead[i] = (i == 0 || skey[i] != skey[i - 1]) ? 1 : 0;
    }
    if (tid == 0) carry = 0;
    __syncthreads();
    // groups: a leader at position i runs to the next leader
    for (int32_t c0 = 0; c0 < ns; c0 += kBwdPlanThreads) {
        const int32_t i = c0 + tid;
        int32_t nk = 0, gcount = 0;
        WlSlice sl{0, 0, 0, 0, 0, 0, 0, 0};
        if (i < ns && lead[i]) {
            sl = slices[sidx[i]];
            nk = sl.k_len > 0 ? (sl.k_len + 127) / 128 : 0;
            gcount = 1;
            while (i + gcount < ns && !lead[i + gcount]) ++gcount;
        }
        int32_t inc = nk;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) warp_tot[w] = inc;
        __syncthreads();
        int32_t base = carry;
        for (int j = 0; j < w; ++j) base += warp_tot[j];
        const int32_t first = base + inc - nk;  // this group's first key tile
        // The warp's groups one after the other, each group's key tiles spread over
        // the 32 lanes (a long document's hundreds of key tiles took one thread
        // most of the plan's time).
        unsigned leaders = __ballot_sync(0xffffffffu, nk > 0);
        while (leaders) {
            const int src = __ffs(leaders) - 1;
            leaders &= leaders - 1;
            const int32_t gi = __shfl_sync(0xffffffffu, i, src);
            const int32_t gfirst = __shfl_sync(0xffffffffu, first, src);
            const int32_t gnk = __shfl_sync(0xffffffffu, nk, src);
            const int32_t gcnt = __shfl_sync(0xffffffffu, gcount, src);
            for (int32_t kt = lane; kt < gnk; kt += 32) {
                int64_t steps = 0;
                for (int32_t m = 0; m < gcnt; ++m) {
                    int32_t qlo, qhi;
                    const WlSlice& sm = slices[sidx[gi + m]];
                    bwd_q_span(sm, kt, qlo, qhi, slice_mask(wl, h, sm, sidx[gi + m]));
                    steps += qhi - qlo;
                }
                for (int32_t g = 0; g < hkv; ++g) {
                    // units of one (group, kv head) are consecutive, key tiles ascending
                    const int32_t uid = gfirst * hkv + g * gnk + kt;
                    if (uid >= bh->cap_units) {
                        atomicCAS(&bh->error, 0, kErrCapacity);
                        continue;
                    }
                    BwdUnit u;
                    u.gbegin = gi;
                    u.gcount = gcnt;
                    u.kt = kt;
                    u.kvh = g;
                    u.cost = (int64_t)G * steps + 1;
                    units[uid] = u;
                    // dynamic: the unit's power-of-two cost class (cost >= 1)
                    const unsigned long long c =
                        dyn ? 1ULL << (63 - __clzll((unsigned long long)u.cost))
                            : (unsigned long long)u.cost;
                    const unsigned long long inv = ((1ULL << kCostBits) - 1) - c;
                    keys[uid] = (inv << kUidBits) | (unsigned long long)uid;
                }
            }
        }
        __syncthreads();
        if (tid == kBwdPlanThreads - 1) carry = base + inc;
        __syncthreads();
    }
    if (tid == 0) bh->nunits = carry * hkv;
}

// ------------------------------------------------------------------ host side
int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Capacities and offsets from bounds; false on invalid arguments.
bool plan_layout(int32_t num_docs, const pva_mask_desc* m, const pva_worklist_params* p,
                 int32_t num_ctas, WlHeader* h) {
    if (!m || !p || num_docs < 0) return false;
    if (p->tile_m <= 0 || p->tile_n <= 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->num_q_heads % p->num_kv_heads != 0 || p->c_tile < 0 || p->refine_iters < 0 ||
        p->refine_iters > 1000 || (p->dispatch != PVA_DISPATCH_DYNAMIC &&
                                   p->dispatch != PVA_DISPATCH_STATIC) ||
        (p->pack_docs != 0 && p->pack_docs != 1) || (p->pack_docs && p->tile_m > 128))
        return false;
    if (num_ctas <= 0 || num_ctas > kMaxBins) return false;
    if (m->q_tokens < 0 || m->k_tokens < 0) return false;
    int64_t cap_segs = 0, cap_slices = 0, max_group = 1, scan_items = num_docs;
    switch (m->kind) {
    case PVA_MASK_CAUSAL:
        cap_segs = cap_slices = num_docs;
        break;
    case PVA_MASK_SLIDING_WINDOW:
        if (m->window < 1) return false;
        cap_segs = cap_slices = num_docs;
        break;
    case PVA_MASK_SHARED_QUESTION:
        if (m->num_prefix_docs < 0 || m->num_prefix_docs > num_docs) return false;
        cap_segs = num_docs;
        cap_slices = (int64_t)num_docs * (m->num_prefix_docs + 1);
        max_group = m->num_prefix_docs + 1;
        break;
    case PVA_MASK_ZIGZAG_PAIR:
        if (m->cp < 1 || m->q_rank < 0 || m->q_rank >= m->cp || m->k_rank < 0 ||
            m->k_rank >= m->cp)
            return false;
        cap_segs = 2 * (int64_t)num_docs;
        cap_slices = 4 * (int64_t)num_docs;
        max_group = 2;
        break;
    case PVA_MASK_ZIGZAG_STEP:
        if (m->cp < 1 || m->ring_step < 0 || m->ring_step >= m->cp ||
            (int64_t)m->cp * num_docs > (INT32_MAX / 8))
            return false;
        if (m->q_tokens != m->k_tokens) return false;
        cap_segs = 2 * (int64_t)m->cp * num_docs;
        cap_slices = 4 * (int64_t)m->cp * num_docs;
        scan_items = (int64_t)m->cp * num_docs;
        max_group = 2;
        break;
    case PVA_MASK_SLICES: {
        if (m->num_slices < 0 || (m->num_slices > 0 && !m->slices)) return false;
        cap_segs = cap_slices = m->num_slices;
        std::vector<std::pair<int32_t, int32_t>> ranges;
        int64_t i = 0;
        max_group = 1;
        while (i < m->num_slices) {
            const pva_slice& a = m->slices[i];
            int64_t j = i;
            while (j < m->num_slices) {
                const pva_slice& b = m->slices[j];
                if (b.q_row0 != a.q_row0 || b.q_len != a.q_len || b.q_pos0 != a.q_pos0) break;
                if (b.q_len < 0 || b.k_len < 0 || b.q_row0 < 0 || b.k_row0 < 0 ||
                    (int64_t)b.q_row0 + b.q_len > m->q_tokens ||
                    (int64_t)b.k_row0 + b.k_len > m->k_tokens ||
                    b.type < PVA_SLICE_FULL || b.type > PVA_SLICE_BI_CAUSAL ||
                    (b.type == PVA_SLICE_BI_CAUSAL && b.window != 0))
                    return false;
                ++j;
            }
            max_group = std::max<int64_t>(max_group, j - i);
            ranges.push_back({a.q_row0, a.q_len});
            i = j;
        }
        std::sort(ranges.begin(), ranges.end());
        for (size_t r = 1; r < ranges.size(); ++r)
            if ((int64_t)ranges[r - 1].first + ranges[r - 1].second > ranges[r].first)
                return false;  // overlapping query segments
        break;
    }
    default:
        return false;
    }
    const int64_t G = p->num_q_heads / p->num_kv_heads;
    const int64_t qt = m->q_tokens / p->tile_m + cap_segs;  // bound on q tiles
    int64_t cap_units = (int64_t)p->num_kv_heads * ((G / 2) * qt + (G % 2) * ((qt + cap_segs + 1) / 2)) + 1;
    int64_t cap_runs = cap_units * max_group;
    if (cap_units >= (1LL << kUidBits) || cap_runs > INT32_MAX || cap_slices > INT32_MAX ||
        cap_segs > INT32_MAX)
        return false;
    memset(h, 0, sizeof *h);
    h->magic = kWlMagic;
    h->version = kWlVersion;
    h->num_ctas = num_ctas;
    h->tile_m = p->tile_m;
    h->tile_n = p->tile_n;
    h->hq = p->num_q_heads;
    h->hkv = p->num_kv_heads;
    h->kind = m->kind;
    h->q_tokens = m->q_tokens;
    h->k_tokens = m->k_tokens;
    h->num_docs = num_docs;
    h->cap_slices = (int32_t)std::max<int64_t>(cap_slices, 1);
    h->cap_segs = (int32_t)std::max<int64_t>(cap_segs, 1);
    h->cap_units = (int32_t)cap_units;
    h->cap_runs = (int32_t)std::max<int64_t>(cap_runs, 1);
    h->c_tile = p->c_tile;
    h->refine_iters = p->refine_iters;
    h->refine_rounds = 0;
    h->dispatch = p->dispatch;
    h->pack_docs =
        p->pack_docs && (m->kind == PVA_MASK_CAUSAL || m->kind == PVA_MASK_SLIDING_WINDOW) ? 1 : 0;
    int64_t o = 256;
    WlOffsets& f = h->off;
    f.slices = o; o = align256(o + (int64_t)h->cap_slices * sizeof(WlSlice));
    f.segs = o; o = align256(o + (int64_t)h->cap_segs * sizeof(WlSeg));
    f.units_enum = o; o = align256(o + cap_units * (int64_t)sizeof(WlUnit));
    f.keys = o; o = align256(o + cap_units * 8);
    f.order = o; o = align256(o + cap_units * 4);
    f.assign = o; o = align256(o + cap_units * 4);
    f.units = o; o = align256(o + cap_units * (int64_t)sizeof(WlUnit));
    f.runs = o; o = align256(o + (int64_t)h->cap_runs * sizeof(WlRun));
    f.cta_off = o; o = align256(o + ((int64_t)num_ctas + 1) * 4);
    f.doc_scan = o; o = align256(o + 6 * (scan_items + 1) * 4);
    f.dorder = o; o = align256(o + cap_units * 4);
    f.cls_work = o; o = align256(o + 64 * 8);
    f.smask = o; o = align256(o + (int64_t)h->cap_slices * 16);
    f.total = o;
    return true;
}

}  // namespace

int32_t resolve_num_ctas(int32_t requested) {
    if (requested > 0) return requested;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

}  // namespace pva

using namespace pva;

extern "C" size_t pva_worklist_bytes(int32_t num_docs, const pva_mask_desc* mask,
                                     const pva_worklist_params* params) {
    if (!params) return 0;
    const int32_t nc = resolve_num_ctas(params->num_ctas);
    WlHeader h;
    if (!plan_layout(num_docs, mask, params, nc, &h)) return 0;
    return (size_t)h.off.total;
}

extern "C" pva_status pva_build_worklist(const int32_t* cu_seqlens_dev, int32_t num_docs,
                                         const pva_mask_desc* mask,
                                         const pva_worklist_params* params, void* worklist_dev,
                                         size_t worklist_bytes, void* stream) {
    if (!mask || !params || !worklist_dev) return PVA_ERR_INVALID_ARG;
    if (mask->kind != PVA_MASK_SLICES && !cu_seqlens_dev) return PVA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(worklist_dev) % 256 != 0) return PVA_ERR_INVALID_ARG;
    const int32_t nc = resolve_num_ctas(params->num_ctas);
    if (nc <= 0) return PVA_ERR_CUDA;
    WlHeader h;
    if (!plan_layout(num_docs, mask, params, nc, &h)) return PVA_ERR_INVALID_ARG;
    if ((int64_t)worklist_bytes < h.off.total) return PVA_ERR_BUFFER_TOO_SMALL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = reinterpret_cast<uint8_t*>(worklist_dev);
    if (mask->kind == PVA_MASK_SLICES && mask->num_slices > 0) {
        // the explicit slice list lives in host memory: copy it, and wait for
        // the copy so that the caller may free its array on return
        static_assert(sizeof(pva_slice) == sizeof(WlSlice), "slice layouts agree");
        if (cudaMemcpyAsync(base + h.off.slices, mask->slices,
                            (size_t)mask->num_slices * sizeof(pva_slice), cudaMemcpyHostToDevice,
                            st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return PVA_ERR_CUDA;
    }
    PlanArgs pa;
    pa.hinit = h;
    pa.base = base;
    pa.cu = cu_seqlens_dev;
    pa.num_docs = num_docs;
    pa.kind = mask->kind;
    pa.window = mask->window;
    pa.num_prefix = mask->num_prefix_docs;
    pa.cp = mask->cp;
    pa.q_rank = mask->q_rank;
    pa.k_rank = mask->k_rank;
    pa.num_slices = mask->num_slices;
    pa.tile_m = params->tile_m;
    pa.hq = params->num_q_heads;
    pa.hkv = params->num_kv_heads;
    pa.q_tokens = mask->q_tokens;
    pa.k_tokens = mask->k_tokens;
    pa.ring_step = mask->ring_step;
    pa.pack_docs = h.pack_docs;
    wl_plan_kernel<<<1, kPlanThreads, 0, st>>>(pa);
    UnitArgs ua{base, params->tile_m, params->tile_n, params->num_q_heads, params->num_kv_heads,
                (long long)params->c_tile};
    const int ub = (h.cap_units + kUnitWarps - 1) / kUnitWarps;
    wl_units_kernel<<<ub, kUnitWarps * 32, 0, st>>>(ua);
    const int sb = (h.cap_units + kSortChunk - 1) / kSortChunk;
    SortArgs sa;
    sa.err = reinterpret_cast<const int32_t*>(base + offsetof(WlHeader, error));
    sa.n = reinterpret_cast<const int32_t*>(base + offsetof(WlHeader, nunits));
    sa.keys = reinterpret_cast<unsigned long long*>(base + h.off.keys);
    sa.order = reinterpret_cast<int32_t*>(base + h.off.order);
    sa.dorder = reinterpret_cast<int32_t*>(base + h.off.dorder);
    sa.cls_work = reinterpret_cast<const unsigned long long*>(base + h.off.cls_work);
    sa.split = reinterpret_cast<int32_t*>(base + offsetof(WlHeader, dispatch_split));
    sa.num_ctas = nc;
    sa.units_enum = reinterpret_cast<const WlUnit*>(base + h.off.units_enum);
    sa.units = reinterpret_cast<WlUnit*>(base + h.off.units);
    if (params->dispatch == PVA_DISPATCH_DYNAMIC) {
        // the CTAs take units at run time in dispatch order: no LPT bins
        wl_sort_chunks_kernel<true><<<sb, kSortThreads, 0, st>>>(sa);
        wl_merge_rank_kernel<kRankDispatch><<<sb, kSortThreads, 0, st>>>(sa);
    } else {
        wl_sort_chunks_kernel<false><<<sb, kSortThreads, 0, st>>>(sa);
        wl_merge_rank_kernel<kRankLpt><<<sb, kSortThreads, 0, st>>>(sa);
        const int bp = ((nc + 31) / 32) * 32;
        const int lpt_f = bp >= 1024 ? 1 : (1024 / bp < 4 ? 1024 / bp : 4);
        wl_lpt_kernel<<<1, bp * lpt_f, 0, st>>>(base, lpt_f);
        wl_sort_chunks_kernel<false><<<sb, kSortThreads, 0, st>>>(sa);
        wl_merge_rank_kernel<kRankCta><<<sb, kSortThreads, 0, st>>>(sa);
    }
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

extern "C" pva_status pva_worklist_error(const void* worklist_dev, int32_t* code_out,
                                         void* stream) {
    if (!worklist_dev || !code_out) return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t code = 0;
    const uint8_t* base = reinterpret_cast<const uint8_t*>(worklist_dev);
    if (cudaMemcpyAsync(&code, base + offsetof(WlHeader, error), 4, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PVA_ERR_CUDA;
    *code_out = code;
    return PVA_OK;
}

extern "C" pva_status pva_worklist_counts(const void* worklist_dev, int64_t* out7, void* stream) {
    if (!worklist_dev || !out7) return PVA_ERR_INVALID_ARG;
    int64_t* out6 = out7;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    WlHeader h;
    if (cudaMemcpyAsync(&h, worklist_dev, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PVA_ERR_CUDA;
    if (h.magic != kWlMagic) return PVA_ERR_INVALID_ARG;
    out6[0] = h.nsegs;
    out6[1] = h.nslices;
    out6[2] = h.nunits;
    out6[3] = h.nruns;
    out6[4] = h.hq > 0 ? (int64_t)(h.pair_sum / (unsigned long long)h.hq) : 0;
    out6[5] = h.hq > 0 ? (int64_t)(h.tile_sum / (unsigned long long)h.hq) : 0;
    out6[6] = h.lpt_steps;
    return h.error ? (h.error >= kErrTimeoutBase ? PVA_ERR_TIMEOUT : PVA_ERR_DEVICE) : PVA_OK;
}

namespace {

constexpr int64_t kFitTileCap = 1LL << 24;  // per-tile cost when pairs carry no time

// Adds one run's per-CTA samples (CTAs that had work) to the sums of the
// two-feature normal equations: pp, uu, pu, pt, ut, tt.
pva_status add_fit_samples(const void* worklist_dev, const uint64_t* cta_busy_ns_dev,
                           cudaStream_t st, double sums[6]) {
    if (!worklist_dev || !cta_busy_ns_dev) return PVA_ERR_INVALID_ARG;
    WlHeader h;
    if (cudaMemcpyAsync(&h, worklist_dev, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PVA_ERR_CUDA;
    // per-CTA samples need the static assignment
    if (h.magic != kWlMagic || h.error != 0 || h.num_ctas <= 0 || h.nunits < 0 ||
        h.dispatch != PVA_DISPATCH_STATIC)
        return PVA_ERR_INVALID_ARG;
    const int32_t B = h.num_ctas, n = h.nunits;
    std::vector<WlUnit> units((size_t)(n > 0 ? n : 1));
    std::vector<uint64_t> busy(2 * (size_t)B);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(worklist_dev);
    if ((n > 0 && cudaMemcpyAsync(units.data(), base + h.off.units, (size_t)n * sizeof(WlUnit),
                                  cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
        cudaMemcpyAsync(busy.data(), cta_busy_ns_dev, busy.size() * sizeof(uint64_t),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return PVA_ERR_CUDA;
    // per CTA: allowed pairs, (sub-tile, kv tile) steps + sub-tiles, busy time
    std::vector<int64_t> P(B, 0), U(B, 0), cntu(B, 0);
    for (int32_t i = 0; i < n; ++i) {
        const WlUnit& u = units[i];
        if (u.cta < 0 || u.cta >= B) return PVA_ERR_INVALID_ARG;
        const int64_t nsub = u.h1 >= 0 ? 2 : 1;
        P[u.cta] += u.pairs;
        U[u.cta] += nsub * ((int64_t)u.ntiles + 1);
        ++cntu[u.cta];
    }
    for (int32_t b = 0; b < B; ++b) {
        if (cntu[b] == 0) continue;  // CTAs without units return at once
        const double t = (double)(busy[2 * b + 1] - busy[2 * b]);
        const double p = (double)P[b], u = (double)U[b];
        sums[0] += p * p;
        sums[1] += u * u;
        sums[2] += p * u;
        sums[3] += p * t;
        sums[4] += u * t;
        sums[5] += t * t;
    }
    return PVA_OK;
}

}  // namespace

extern "C" pva_status pva_fit_tile_cost(const void* const* worklists_dev,
                                        const uint64_t* const* cta_busy_ns_dev, int32_t num_runs,
                                        int64_t* c_tile_out, double* coef_out, void* stream) {
    if (!worklists_dev || !cta_busy_ns_dev || !c_tile_out || num_runs <= 0)
        return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    double sm[6] = {0, 0, 0, 0, 0, 0};
    for (int32_t r = 0; r < num_runs; ++r) {
        const pva_status s = add_fit_samples(worklists_dev[r], cta_busy_ns_dev[r], st, sm);
        if (s != PVA_OK) return s;
    }
    const double pp = sm[0], uu = sm[1], pu = sm[2], pt = sm[3], ut = sm[4], tt = sm[5];
    // non-negative least squares in two unknowns: the unconstrained solution if
    // feasible, else the better of the two one-feature fits
    double a = 0, c = 0;
    const double det = pp * uu - pu * pu;
    bool ok = false;
    if (det > 0) {
        a = (pt * uu - pu * ut) / det;
        c = (pp * ut - pu * pt) / det;
        ok = a >= 0 && c >= 0;
    }
    if (!ok) {
        const double a1 = pp > 0 && pt > 0 ? pt / pp : 0, c1 = uu > 0 && ut > 0 ? ut / uu : 0;
        const double r_a = tt - 2 * a1 * pt + a1 * a1 * pp;
        const double r_c = tt - 2 * c1 * ut + c1 * c1 * uu;
        if (r_a <= r_c) {
            a = a1;
            c = 0;
        } else {
            a = 0;
            c = c1;
        }
    }
    if (coef_out) {
        coef_out[0] = a;
        coef_out[1] = c;
    }
    if (a > 0) {
        const double r = c / a;
        *c_tile_out = r >= (double)kFitTileCap ? kFitTileCap : (int64_t)std::llround(r);
        return PVA_OK;
    }
    if (c > 0) {
        *c_tile_out = kFitTileCap;
        return PVA_OK;
    }
    return PVA_ERR_INVALID_ARG;
}

namespace {

bool bwd_layout(int32_t num_docs, const pva_mask_desc* mask, const pva_worklist_params* params,
                BwdHeader* bh) {
    if (!mask || !params) return false;
    // slices' key ranges must be identical or disjoint: a key group then owns
    // its key rows (the built-in mask kinds satisfy this by construction)
    if (mask->kind == PVA_MASK_SLICES) {
        if (!mask->slices || mask->num_slices < 0) return false;
        std::vector<std::pair<int32_t, int32_t>> kr;
        for (int32_t i = 0; i < mask->num_slices; ++i)
            if (mask->slices[i].k_len > 0)
                kr.push_back({mask->slices[i].k_row0, mask->slices[i].k_row0 + mask->slices[i].k_len});
        std::sort(kr.begin(), kr.end());
        kr.erase(std::unique(kr.begin(), kr.end()), kr.end());
        for (size_t i = 1; i < kr.size(); ++i)
            if (kr[i].first < kr[i - 1].second) return false;
    }
    WlHeader h;
    const int32_t nc = resolve_num_ctas(params->num_ctas);
    if (nc <= 0 || !plan_layout(num_docs, mask, params, nc, &h)) return false;
    if (h.cap_slices > kBwdMaxSlices) return false;
    const int64_t hkv = params->num_kv_heads;
    const int64_t cap = ((int64_t)(mask->k_tokens + 127) / 128 + h.cap_slices) * hkv + 1;
    if (cap >= (1LL << kUidBits)) return false;
    memset(bh, 0, sizeof *bh);
    bh->magic = kBwdMagic;
    bh->cap_units = (int32_t)cap;
    bh->hq = params->num_q_heads;
    bh->hkv = params->num_kv_heads;
    bh->q_tokens = mask->q_tokens;
    bh->k_tokens = mask->k_tokens;
    int64_t o = 256;
    bh->off_units = o; o = align256(o + cap * (int64_t)sizeof(BwdUnit));
    bh->off_keys = o; o = align256(o + cap * 8);
    bh->off_order = o; o = align256(o + cap * 4);
    bh->off_gslices = o; o = align256(o + (int64_t)h.cap_slices * 4 + 4);
    bh->off_dvec = o; o = align256(o + (int64_t)params->num_q_heads * mask->q_tokens * 4);
    bh->total = o;
    return true;
}

}  // namespace

namespace pva {
int64_t bwd_plan_dvec_offset(int32_t num_docs, const pva_mask_desc* mask,
                             const pva_worklist_params* params) {
    BwdHeader bh;
    if (!bwd_layout(num_docs, mask, params, &bh)) return -1;
    return bh.off_dvec;
}
}  // namespace pva

extern "C" size_t pva_bwd_plan_bytes(int32_t num_docs, const pva_mask_desc* mask,
                                     const pva_worklist_params* params) {
    BwdHeader bh;
    if (!bwd_layout(num_docs, mask, params, &bh)) return 0;
    return (size_t)bh.total;
}

extern "C" pva_status pva_build_bwd_plan(const void* worklist_dev, int32_t num_docs,
                                         const pva_mask_desc* mask,
                                         const pva_worklist_params* params, void* plan_dev,
                                         size_t plan_bytes, void* stream) {
    if (!worklist_dev || !plan_dev || (reinterpret_cast<uintptr_t>(plan_dev) & 255u))
        return PVA_ERR_INVALID_ARG;
    BwdHeader bh;
    if (!bwd_layout(num_docs, mask, params, &bh)) return PVA_ERR_INVALID_ARG;
    if (plan_bytes < (size_t)bh.total) return PVA_ERR_BUFFER_TOO_SMALL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = reinterpret_cast<uint8_t*>(plan_dev);
    if (cudaMemcpyAsync(base, &bh, sizeof bh, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return PVA_ERR_CUDA;
    // shared memory: sort keys, slice indices and group flags for every slice
    const size_t smem = (size_t)kBwdMaxSlices * 16;
    if (cudaFuncSetAttribute(bwd_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return PVA_ERR_CUDA;
    bwd_plan_kernel<<<1, kBwdPlanThreads, smem, st>>>(
        reinterpret_cast<const uint8_t*>(worklist_dev), base);
    SortArgs sa;
    sa.err = reinterpret_cast<const int32_t*>(base + offsetof(BwdHeader, error));
    sa.n = reinterpret_cast<const int32_t*>(base + offsetof(BwdHeader, nunits));
    sa.keys = reinterpret_cast<unsigned long long*>(base + bh.off_keys);
    sa.order = reinterpret_cast<int32_t*>(base + bh.off_order);
    sa.dorder = nullptr;
    sa.cls_work = nullptr;
    sa.split = nullptr;
    sa.num_ctas = 0;
    sa.units_enum = nullptr;
    sa.units = nullptr;
    const int sb = (bh.cap_units + kSortChunk - 1) / kSortChunk;
    wl_sort_chunks_kernel<false><<<sb, kSortThreads, 0, st>>>(sa);
    wl_merge_rank_kernel<kRankLpt><<<sb, kSortThreads, 0, st>>>(sa);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}
