// attn_bwd.cu -- backward of the packed document-masked attention on sm_103a.
//
// The gradients of the quadratic term of "03 · 长文负载均衡" §1.1 (QK^T and
// PV) over the same AttnSlices as the forward.  With P = exp(scale S - LSE)
// recomputed from the forward's LSE:
//   dP = dO V^T,  D = rowsum(dO * O),  dS = P (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// Three kernels, no atomics (each output row has one writer):
//   bwd_pre   D per (row, head), HBM-bound;
//   bwd_dq    q-major over the forward worklist's units, dispatched as the
//             worklist says (static per-CTA LPT lists, or claimed at run time):
//             per query sub-tile (Q and dO copied into tensor memory), every
//             kv tile of its runs as two 64-key halves: S and dP (TS MMAs,
//             issued by two warps), then dS in the element-wise warps, then
//             dQ += dS K (TS MMA);
//   bwd_dkdv  kv-major over the backward plan: per 128-key tile of one key
//             group (the slices sharing a key range) and one kv head, every q
//             tile of every slice of the group, each for every head of the kv
//             head's group (a q tile's heads back to back): S^T = K Q^T and
//             dP^T = V dO^T, then P^T and dS^T, then dV += P^T dO and
//             dK += dS^T Q, accumulated in tensor memory over the group; a
//             loader warp stages each 64-query half's LSE and D ahead.
// In both passes two element-wise warpgroups share every half-item (32
// columns each) so that its P / dS are ready as early as possible.
// Tensor-memory columns: bwd_dq S [0,128) dP [128,256) dQ [256,256+d), then Q and
// dO as bf16 MMA A operands (d/2 columns each);
// bwd_dkdv with nb S^T / dP^T buffers (2 at d = 128, 3 at d = 64): S^T [0,64 nb)
// dP^T [64 nb,128 nb) dV [128 nb,128 nb+d) dK [128 nb+d,128 nb+2d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/pva.h"
#include "common.h"
#include "ptx.cuh"
#include "tma_map.h"
#include "unit_feed.cuh"
#include "wl_layout.cuh"

namespace pva {
namespace {

// warp 0 TMA, warp 1 MMA (bwd_dq: warp 3 issues its dP MMAs), warp 2 the dK/dV
// pass's (LSE, D) loader, warps 4-11 element-wise + epilogue (two warpgroups
// sharing every half-item)
constexpr int kThreads = 384;
// bwd_dkdv's register split (kSplitRegs): the TMA/MMA warpgroup gives registers
// to the two element-wise warpgroups
constexpr bool kSplitRegs = false;
constexpr uint32_t kRegsCtrl = 152, kRegsElem = 176;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

template <int D>
struct BCfg {
    static constexpr int kTileBytes = 128 * D * 2;
    // bwd_dq: Q, dO, then a K/V ring; bwd_dkdv: K, V, then a (Q, dO) ring
    // ring stages: as many as fit beside the two resident tiles within 227 KB of
    // shared memory per block (bwd_dkdv also holds 2.3 KB of static staging)
    static constexpr int kStagesDq = D == 128 ? 5 : 12;
    static constexpr int kStagesKv = D == 128 ? 4 : 11;
    // bwd_dkdv's S^T / dP^T buffers (64 + 64 tensor-memory columns each): d = 64
    // leaves room for a third beside dV and dK
    static constexpr uint32_t kBufsKv = D == 64 ? 3 : 2;  // at most 3
    static constexpr int kSmemDq = 2 * kTileBytes + kStagesDq * kTileBytes + 1024;
    static constexpr int kSmemKv = 2 * kTileBytes + kStagesKv * kTileBytes + 1024;
    static constexpr uint32_t kIdescNN = idesc_bf16_f32(128, D, true);     // B MN-major
};

struct BwdParams {
    const uint8_t* wl;
    const uint8_t* plan;
    const void* out;     // forward output O, bf16 [Tq, Hq, d]
    const void* dout;    // dO, bf16 [Tq, Hq, d]
    const float* lse;    // forward LSE (natural log) [Hq, Tq]
    float* dvec;         // D [Hq, Tq]
    void* dq;            // [Tq, Hq, d]
    void* dk;            // [Tk, Hkv, d]
    void* dv;            // [Tk, Hkv, d]
    int32_t q_tokens, k_tokens, hq, hkv, grads_fp32, num_ctas, d;
    float scale, scale_log2;
};

constexpr int kLdSlots = 8;
constexpr int kMaxStages = 12;

struct BShared {
    uint64_t a_full, a_empty, o_full, o_empty, done, done2;
    uint64_t s2_full[3], p2_full[3];  // per half-item tensor-memory buffer
    uint64_t r_full[kMaxStages], r_empty[kMaxStages];
    UnitRing<8> ur;  // the producer hands each unit's index to the other roles
    // bwd_dkdv: (LSE log2, D) of each half-item's 64 queries, staged ahead by a
    // loader warp (ld_full: 32 lane arrivals; ld_empty: one per element-wise warp)
    uint64_t ld_full[kLdSlots], ld_empty[kLdSlots];
    uint32_t tmem_base;
    int32_t abort_flag;
};

// ------------------------------------------------------------ D = rowsum(dO O)
// 8 threads per (row, head), 16 bytes each per step.
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdParams p) {
    const int64_t rows = (int64_t)p.q_tokens * p.hq;
    const int sub = threadIdx.x & 7;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 3;
         r - (threadIdx.x & 31) / 8 < rows; r += ((int64_t)gridDim.x * blockDim.x) >> 3) {
        float acc = 0.f;
        if (r < rows) {
            const uint4* o = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.out) + r * p.d);
            const uint4* g = reinterpret_cast<const uint4*>(
                reinterpret_cast<const __nv_bfloat16*>(p.dout) + r * p.d);
            for (int c = sub; c < p.d / 8; c += 8) {
                const uint4 a = o[c], b = g[c];
                const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
                    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[e]));
                    acc += fa.x * fb.x + fa.y * fb.y;
                }
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (r < rows && sub == 0) {
            const int64_t t = r / p.hq;
            const int32_t h = (int32_t)(r - t * p.hq);
            p.dvec[(int64_t)h * p.q_tokens + t] = acc;
        }
    }
}

// Writes 32 fp32 accumulator columns of one row, scaled, as fp32 or bf16.
__device__ __forceinline__ void store_row32(void* base, int64_t row_elem, bool fp32,
                                            const uint32_t (&v)[32], float scale) {
    if (fp32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + row_elem);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(v[4 * e]) * scale, __uint_as_float(v[4 * e + 1]) * scale,
                                 __uint_as_float(v[4 * e + 2]) * scale,
                                 __uint_as_float(v[4 * e + 3]) * scale);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + row_elem);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * e]) * scale, __uint_as_float(v[8 * e + 1]) * scale),
                pack_bf16x2(__uint_as_float(v[8 * e + 2]) * scale, __uint_as_float(v[8 * e + 3]) * scale),
                pack_bf16x2(__uint_as_float(v[8 * e + 4]) * scale, __uint_as_float(v[8 * e + 5]) * scale),
                pack_bf16x2(__uint_as_float(v[8 * e + 6]) * scale, __uint_as_float(v[8 * e + 7]) * scale));
    }
}

// The element-wise warpgroup c (0, 1) turns the 32 fp32 columns [32c, 32c + 32)
// of a 64-column S / dP buffer into 32 bf16 values packed in its first 16
// columns, so the warpgroups never overwrite columns the other still reads.
// The 16-wide K slice k of that bf16 operand therefore starts at column:
__device__ __forceinline__ uint32_t kslice_col(int k) { return (k >> 1) * 32 + (k & 1) * 8; }

__device__ __forceinline__ void store_zero_row(void* base, int64_t row_elem, bool fp32, int D) {
    if (fp32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + row_elem);
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + row_elem);
        for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    }
}

// issuers: MMA-issuing warps; each commits once to a_empty, s2_full and r_empty
// per use and reads every unit.  acc_issuers: the warps that commit o_full (the
// ones whose MMAs write the accumulators).  item_warps: the element-wise warps
// that work on each half-item (p2_full and ld_empty count one arrival each)
__device__ __forceinline__ void init_barriers(BShared& sh, int stages, int elem_threads,
                                              int extra_readers, int issuers, int acc_issuers,
                                              int item_warps) {
    mbar_init(&sh.a_full, 1);
    mbar_init(&sh.a_empty, issuers);
    mbar_init(&sh.o_full, acc_issuers);
    mbar_init(&sh.o_empty, elem_threads / 32);
    mbar_init(&sh.done, 1);
    mbar_init(&sh.done2, 1);
    for (int b = 0; b < 3; ++b) {
        mbar_init(&sh.s2_full[b], issuers);
        mbar_init(&sh.p2_full[b], item_warps);
    }
    for (int s = 0; s < stages; ++s) {
        mbar_init(&sh.r_full[s], 1);
        mbar_init(&sh.r_empty[s], issuers);
    }
    // unit readers: the MMA warps (one arrival each) and every element-wise thread
    uring_init(sh.ur, issuers + elem_threads + extra_readers);
    for (int s = 0; s < kLdSlots; ++s) {
        mbar_init(&sh.ld_full[s], 32);
        mbar_init(&sh.ld_empty[s], item_warps);
    }
    sh.abort_flag = 0;
    fence_barrier_init();
}

// ==================================================================== dQ
// Per query sub-tile (forward worklist units, sub-tiles one after the other):
// a_full/a_empty guard the Q and dO tiles; the keys stream as half-items (64
// keys [64 hf, 64 hf + 64) of a kv tile: K and V halves, 64-row TMA boxes)
// through a ring (r_full/r_empty).  S and dP of half-item u (N = 64) go to one
// of two 64-column buffers (s2_full/p2_full) and are issued before dQ += dS K
// of half-item u - 1, so dS of u - 1 is computed while the pipe works on u.
// o_full/o_empty: dQ accumulated / read out.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                  const BwdParams p) {
    // tmk and tmv have 64-row boxes here (key half-items)
    using C = BCfg<D>;
    constexpr int kHalfBytes = 64 * D * 2;  // one 64-row bf16 half tile; a stage holds K and V halves
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sDO = smem + C::kTileBytes;
    uint8_t* sKV = smem + 2 * C::kTileBytes;
    __shared__ BShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WlHeader* h = reinterpret_cast<const WlHeader*>(p.wl);
    int32_t* err_word = const_cast<int32_t*>(&h->error);
    if (h->error != 0) return;
    // the worklist's dispatch: static per-CTA lists of `units`, or (dynamic)
    // ranks of `dorder` claimed at run time from the worklist's counter
    const bool dyn = h->dispatch == PVA_DISPATCH_DYNAMIC;
    WlHeader* hw = const_cast<WlHeader*>(h);
    const int32_t nunits = h->nunits;
    const int32_t* dorder = reinterpret_cast<const int32_t*>(p.wl + h->off.dorder);
    const WlUnit* ubase = reinterpret_cast<const WlUnit*>(p.wl + (dyn ? h->off.units_enum
                                                                       : h->off.units));
    const WlRun* runs = reinterpret_cast<const WlRun*>(p.wl + h->off.runs);
    const WlSlice* slices = reinterpret_cast<const WlSlice*>(p.wl + h->off.slices);
    const WlSeg* segs = reinterpret_cast<const WlSeg*>(p.wl + h->off.segs);
    const int32_t* cta_off = reinterpret_cast<const int32_t*>(p.wl + h->off.cta_off);
    const int32_t ub = dyn ? 0 : cta_off[blockIdx.x], ue = dyn ? 0 : cta_off[blockIdx.x + 1];
    if (!dyn && ub >= ue) return;
    if (tid == 0) init_barriers(sh, C::kStagesDq, 256, 0, 2, 1, 8);
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmdo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int32_t* abort_flag = &sh.abort_flag;

    // the two query sub-tiles of a unit, one after the other
    auto sub_of = [&](const WlUnit& u, int i, int32_t& q_row, int32_t& nrows, int32_t& q_pos,
                      int32_t& head) {
        const WlSeg g = segs[u.seg];
        const int32_t t = i == 0 ? u.t0 : u.t1;
        q_row = g.q_row0 + t * 128;
        nrows = min(128, g.q_len - t * 128);
        q_pos = g.q_pos0 + t * 128;
        head = i == 0 ? u.h0 : u.h1;
    };

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, a_it = 0;
            bool live = true;
            for (uint32_t nu = 0; live; ++nu) {
                live = uring_wait_free(sh.ur, nu, abort_flag, err_word, kErrTimeoutBase + 29,
                                       kWaitNs);
                if (!live) break;
                int32_t idx;
                if (dyn) {
                    const int32_t rank = dispatch_claim(&hw->dispatch_next);
                    idx = rank < nunits ? dorder[rank] : -1;
                    if (idx >= nunits || idx < -1) {  // a damaged order: stop, report
                        atomicCAS(err_word, 0, kErrBadWorklist);
                        idx = -1;
                    }
                } else {
                    idx = ub + (int32_t)nu < ue ? ub + (int32_t)nu : -1;
                }
                uring_put(sh.ur, nu, idx);
                if (idx < 0) break;
                const WlUnit u = ubase[idx];
                if (u.ntiles == 0) continue;
                const int nsub = u.h1 >= 0 ? 2 : 1;
                for (int i = 0; i < nsub && live; ++i) {
                    int32_t q_row, nrows, q_pos, head;
                    sub_of(u, i, q_row, nrows, q_pos, head);
                    live = mbar_wait(&sh.a_empty, (a_it & 1) ^ 1, abort_flag, err_word,
                                     kErrTimeoutBase + 21, kWaitNs);
                    if (!live) break;
                    mbar_arrive_expect_tx(&sh.a_full, 2 * C::kTileBytes);
                    for (int b = 0; b < D / 64; ++b) {
                        tma_load_3d(sQ + b * 16384, &tmq, &sh.a_full, b * 64, head, q_row);
                        tma_load_3d(sDO + b * 16384, &tmdo, &sh.a_full, b * 64, head, q_row);
                    }
                    ++a_it;
                    for (int32_t rr = 0; rr < u.run_count && live; ++rr) {
                        const WlRun run = runs[u.run_begin + rr];
                        const WlSlice s = slices[run.slice];
                        for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                            const int32_t halves = min(128, s.k_len - jt * 128) > 64 ? 2 : 1;
                            for (int32_t hf = 0; hf < halves && live; ++hf) {
                                const int32_t krow = s.k_row0 + jt * 128 + hf * 64;
                                const uint32_t st = it % C::kStagesDq;
                                live = mbar_wait(&sh.r_empty[st], ((it / C::kStagesDq) & 1) ^ 1,
                                                 abort_flag, err_word, kErrTimeoutBase + 22,
                                                 kWaitNs);
                                if (!live) break;
                                mbar_arrive_expect_tx(&sh.r_full[st], 2 * kHalfBytes);
                                uint8_t* dk_ = sKV + st * 2 * kHalfBytes;
                                for (int b = 0; b < D / 64; ++b) {
                                    tma_load_3d(dk_ + b * 8192, &tmk, &sh.r_full[st], b * 64,
                                                u.kvh, krow);
                                    tma_load_3d(dk_ + kHalfBytes + b * 8192, &tmv, &sh.r_full[st],
                                                b * 64, u.kvh, krow);
                                }
                                ++it;
                            }
                        }
                    }
                }
            }
            if (!live) {
                const uint32_t n = it < (uint32_t)C::kStagesDq ? it : (uint32_t)C::kStagesDq;
                for (uint32_t k = 0; k < n; ++k) {
                    const uint32_t x = it - 1 - k;
                    mbar_wait_drain(&sh.r_full[x % C::kStagesDq], (x / C::kStagesDq) & 1, kDrainNs);
                }
                if (a_it > 0) mbar_wait_drain(&sh.a_full, (a_it - 1) & 1, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer (whole warp)
        uint32_t it = 0, a_it = 0, gu = 0, o_cnt = 0;
        bool live = true;
        const uint64_t dQd = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dKn = sdesc_sw128(smem_u32(sKV), 16, 1024);    // K-major, 64-row atoms
        const uint64_t dKm = sdesc_sw128(smem_u32(sKV), 8192, 1024);  // MN-major, 64-row atoms
        constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, false);
        const uint32_t tQa = tmem + 256;
        // Q and dO of the sub-tile, copied into tensor memory as the A operands of
        // S = Q K^T and dP = dO V^T (TS MMAs read only the K / V halves from shared
        // memory, so N = 64 runs at the full rate)
        const uint32_t tQA = tmem + 256 + D;
        bool pend = false, first = true;
        uint32_t pend_u = 0, pend_st = 0;
        auto finish_pending = [&]() -> bool {
            const uint32_t b = pend_u & 1;
            // the sub-tile's first dQ MMA overwrites the accumulator: the previous
            // sub-tile's epilogue must have read it (waited only here, so that S and
            // dP of the first half-items overlap that epilogue)
            if (first && !mbar_wait_warp(&sh.o_empty, (o_cnt & 1) ^ 1, abort_flag, err_word,
                                         kErrTimeoutBase + 24, kWaitNs))
                return false;
            if (!mbar_wait_warp(&sh.p2_full[b], (pend_u >> 1) & 1, abort_flag, err_word,
                                kErrTimeoutBase + 26, kWaitNs))
                return false;
            tc_fence_after();
            const uint64_t oK = (pend_st * 2 * kHalfBytes) >> 4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_ts_elect(tQa, tmem + 64 * b + kslice_col(k), dKm + oK + k * 128, C::kIdescNN,
                             (!first || k > 0) ? 1u : 0u);
            first = false;
            mma_commit_elect(&sh.r_empty[pend_st]);
            pend = false;
            return true;
        };
        for (uint32_t nu = 0; live; ++nu) {
            int32_t idx;
            live = uring_get_warp(sh.ur, nu, idx, abort_flag, err_word, kErrTimeoutBase + 30,
                                  kWaitNs);
            if (!live || idx < 0) break;
            const WlUnit u = ubase[idx];
            if (u.ntiles == 0) continue;
            const int nsub = u.h1 >= 0 ? 2 : 1;
            for (int i = 0; i < nsub && live; ++i) {
                live = mbar_wait_warp(&sh.a_full, a_it & 1, abort_flag, err_word,
                                      kErrTimeoutBase + 23, kWaitNs);
                if (!live) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off16 = (k >> 2) * 1024 + (k & 3) * 2;
                    tmem_cp_elect(tQA + k * 8, dQd + off16);
                }
                mma_commit_elect(&sh.a_empty);  // Q copied (warp 3 copies dO)
                first = true;
                for (int32_t rr = 0; rr < u.run_count && live; ++rr) {
                    const WlRun run = runs[u.run_begin + rr];
                    const WlSlice s = slices[run.slice];
                    for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                        const int32_t halves = min(128, s.k_len - jt * 128) > 64 ? 2 : 1;
                        for (int32_t hf = 0; hf < halves && live; ++hf) {
                            const uint32_t st = it % C::kStagesDq;
                            live = mbar_wait_warp(&sh.r_full[st], (it / C::kStagesDq) & 1,
                                                  abort_flag, err_word, kErrTimeoutBase + 25,
                                                  kWaitNs);
                            if (!live) break;
                            tc_fence_after();
                            const uint32_t b = gu & 1;
                            const uint64_t oK = (st * 2 * kHalfBytes) >> 4;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                // Q (tensor memory) against the K half (64-row atoms)
                                const uint32_t kq = (k >> 2) * 512 + (k & 3) * 2;
                                mma_ts_elect(tmem + 64 * b, tQA + k * 8, dKn + oK + kq, kIdescHalf,
                                             k > 0);
                            }
                            mma_commit_elect(&sh.s2_full[b]);
                            if (pend && !finish_pending()) {
                                live = false;
                                break;
                            }
                            pend = true;
                            pend_u = gu;
                            pend_st = st;
                            ++gu;
                            ++it;
                        }
                    }
                }
                if (!live) break;
                if (pend && !finish_pending()) break;
                mma_commit_elect(&sh.o_full);
                ++o_cnt;
                ++a_it;
            }
        }
        mma_commit_elect(&sh.done);
        mbar_wait_drain(&sh.done, 0, kDrainNs);
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------- dP issuer (whole warp)
        // dP = dO V^T of every half-item into buffer b = half-item % 2, from a warp
        // of its own: one issuing warp spends about as long issuing a half-item's
        // 20 MMAs as the tensor pipe takes to run them.  The dP buffer is reused
        // once the element-wise warps have read it (p2_full of two half-items ago);
        // the stage is released by both issuers (r_empty counts two commits).
        uint32_t it = 0, a_it = 0, gu = 0;
        bool live = true;
        const uint64_t dDO = sdesc_sw128(smem_u32(sDO), 16, 1024);
        const uint64_t dKn = sdesc_sw128(smem_u32(sKV), 16, 1024);  // K-major, 64-row atoms
        constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, false);
        const uint32_t tDOA = tmem + 256 + D + D / 2;
        for (uint32_t nu = 0; live; ++nu) {
            int32_t idx;
            live = uring_get_warp(sh.ur, nu, idx, abort_flag, err_word, kErrTimeoutBase + 46,
                                  kWaitNs);
            if (!live || idx < 0) break;
            const WlUnit u = ubase[idx];
            if (u.ntiles == 0) continue;
            const int nsub = u.h1 >= 0 ? 2 : 1;
            for (int i = 0; i < nsub && live; ++i) {
                live = mbar_wait_warp(&sh.a_full, a_it & 1, abort_flag, err_word,
                                      kErrTimeoutBase + 47, kWaitNs);
                if (!live) break;
                tc_fence_after();
                // dO of the sub-tile into tensor memory (after this warp's last dP of
                // the previous sub-tile, in issue order)
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    tmem_cp_elect(tDOA + k * 8, dDO + (k >> 2) * 1024 + (k & 3) * 2);
                mma_commit_elect(&sh.a_empty);
                for (int32_t rr = 0; rr < u.run_count && live; ++rr) {
                    const WlRun run = runs[u.run_begin + rr];
                    const WlSlice s = slices[run.slice];
                    for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                        const int32_t halves = min(128, s.k_len - jt * 128) > 64 ? 2 : 1;
                        for (int32_t hf = 0; hf < halves && live; ++hf) {
                            const uint32_t st = it % C::kStagesDq;
                            const uint32_t b = gu & 1;
                            live = mbar_wait_warp(&sh.r_full[st], (it / C::kStagesDq) & 1,
                                                  abort_flag, err_word, kErrTimeoutBase + 48,
                                                  kWaitNs);
                            if (!live) break;
                            if (gu >= 2) {
                                live = mbar_wait_warp(&sh.p2_full[b], ((gu - 2) >> 1) & 1,
                                                      abort_flag, err_word, kErrTimeoutBase + 49,
                                                      kWaitNs);
                                if (!live) break;
                            }
                            tc_fence_after();
                            const uint64_t oV = (st * 2 * kHalfBytes + kHalfBytes) >> 4;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint32_t kq = (k >> 2) * 512 + (k & 3) * 2;
                                mma_ts_elect(tmem + 128 + 64 * b, tDOA + k * 8, dKn + oV + kq,
                                             kIdescHalf, k > 0);
                            }
                            mma_commit_elect(&sh.s2_full[b]);
                            mma_commit_elect(&sh.r_empty[st]);
                            ++gu;
                            ++it;
                        }
                    }
                }
                if (!live) break;
                ++a_it;
            }
        }
        mma_commit_elect(&sh.done2);
        mbar_wait_drain(&sh.done2, 0, kDrainNs);
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------- dS and the dQ epilogue
        // Two warpgroups share every half-item: wg takes its 32 key columns
        // [32 wg, 32 wg + 32), so a half-item's dS is ready in half the time;
        // each stores half of the dQ columns.
        const int wg = (warp - 4) >> 2;
        const int r = (warp & 3) * 32 + lane;  // query row = tensor-memory lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base, tQ = tmem + lane_base + 256;
        uint32_t gu = 0, o_cnt = 0;
        bool live = true;
        for (uint32_t nu = 0; live; ++nu) {
            int32_t idx;
            live = uring_get(sh.ur, nu, idx, abort_flag, err_word, kErrTimeoutBase + 30, kWaitNs);
            if (!live || idx < 0) break;
            const WlUnit u = ubase[idx];
            const int nsub = u.h1 >= 0 ? 2 : 1;
            for (int i = 0; i < nsub && live; ++i) {
                int32_t q_row, nrows, q_pos0, head;
                sub_of(u, i, q_row, nrows, q_pos0, head);
                const bool valid = r < nrows;
                const int64_t grow = ((int64_t)(q_row + r) * p.hq + head) * D;
                if (u.ntiles == 0) {  // rows without keys: zero gradient
                    if (valid) store_zero_row(p.dq, grow + wg * (D / 2), p.grads_fp32, D / 2);
                    continue;
                }
                const int32_t q_pos = q_pos0 + r;
                const int64_t li = (int64_t)head * p.q_tokens + q_row + r;
                float lse2 = INFINITY, dd = 0.f;  // no key: every P is 0
                if (valid) {
                    const float l = p.lse[li];
                    if (l != -INFINITY) lse2 = l * 1.4426950408889634f;
                    dd = p.dvec[li];
                }
                for (int32_t rr = 0; rr < u.run_count && live; ++rr) {
                    const WlRun run = runs[u.run_begin + rr];
                    const WlSlice s = slices[run.slice];
                    int64_t klo, khi;  // allowed keys of this row (slice-local)
                    slice_keys_of_query(s, q_pos, klo, khi, slice_mask(p.wl, h, s, run.slice));
                    const int32_t lim_hi = valid ? (int32_t)khi : 0;
                    const int32_t lim_lo = (int32_t)klo;
                    for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                        const int32_t kt0 = jt * 128;
                        const int32_t c_hi = min(128, lim_hi - kt0), c_lo = max(0, lim_lo - kt0);
                        const int32_t halves = min(128, s.k_len - kt0) > 64 ? 2 : 1;
                        for (int32_t hf = 0; hf < halves && live; ++hf, ++gu) {
                            const uint32_t b = gu & 1;
                            // this warpgroup's 32 key columns [h0, h0 + 32) of the half; the
                            // warp masks only when some row has a limit inside them
                            const int h0 = hf * 64 + wg * 32;
                            const bool need_mask =
                                __any_sync(0xffffffffu, c_lo > h0 || c_hi < h0 + 32);
                            live = mbar_wait(&sh.s2_full[b], (gu >> 1) & 1, abort_flag, err_word,
                                             kErrTimeoutBase + 27, kWaitNs);
                            if (!live) break;
                            tc_fence_after();
                            const uint32_t tSb = tS + 64 * b, tPb = tS + 128 + 64 * b;
                            {
                                const int c = wg;
                                uint32_t sv[32], pv[32];
                                tmem_ld32(tSb + c * 32, sv);
                                tmem_ld32(tPb + c * 32, pv);
                                tmem_ld_wait(sv);
                                tmem_ld_wait(pv);
                                uint32_t dsw[32];
                                const float2 sc = make_float2(p.scale_log2, p.scale_log2);
                                const float2 nl = make_float2(-lse2, -lse2);
                                const float2 nd = make_float2(-dd, -dd);
#pragma unroll
                                for (int e = 0; e < 32; e += 2) {
                                    const int col = hf * 64 + c * 32 + e;
                                    const float2 x =
                                        __ffma2_rn(make_float2(__uint_as_float(sv[e]),
                                                               __uint_as_float(sv[e + 1])),
                                                   sc, nl);
                                    float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                                    if (need_mask) {
                                        if (col < c_lo || col >= c_hi) p0 = 0.f;
                                        if (col + 1 < c_lo || col + 1 >= c_hi) p1 = 0.f;
                                    }
                                    const float2 g = __fmul2_rn(
                                        make_float2(p0, p1),
                                        __fadd2_rn(make_float2(__uint_as_float(pv[e]),
                                                               __uint_as_float(pv[e + 1])),
                                                   nd));
                                    dsw[e >> 1] = pack_bf16x2(g.x, g.y);
                                }
                                tmem_st16(tSb + c * 32, dsw);
                            }
                            tmem_st_wait();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.p2_full[b]);
                        }
                    }
                }
                if (!live) break;
                live = mbar_wait(&sh.o_full, o_cnt & 1, abort_flag, err_word,
                                 kErrTimeoutBase + 28, kWaitNs);
                if (!live) break;
                ++o_cnt;
                tc_fence_after();
                // this warpgroup's half of the dQ columns
                constexpr int kHalfChunks = D / 64;
                uint32_t o[kHalfChunks][32];
#pragma unroll
                for (int c = 0; c < kHalfChunks; ++c)
                    tmem_ld32(tQ + (wg * kHalfChunks + c) * 32, o[c]);
#pragma unroll
                for (int c = 0; c < kHalfChunks; ++c) tmem_ld_wait(o[c]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.o_empty);
                if (valid) {
#pragma unroll
                    for (int c = 0; c < kHalfChunks; ++c)
                        store_row32(p.dq, grow + (wg * kHalfChunks + c) * 32, p.grads_fp32, o[c],
                                    p.scale);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (dyn && tid == 0) dispatch_exit(&hw->dispatch_next, &hw->dispatch_done);
}

// ==================================================================== dK, dV
// Per backward-plan unit (128 keys of one slice, one kv head): K and V stay in
// shared memory (a_full/a_empty), the (Q, dO) tiles of every (head, q tile)
// item stream through a ring of item pairs (r_full/r_empty per item).
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ CUtensorMap tmdo, const BwdParams p) {
    // tmq and tmdo have 64-row boxes here: the ring holds half-items, the 64
    // queries [64 hf, 64 hf + 64) of a q tile as (Q, dO) halves of 8 KB per
    // 64-column atom (a stage: Q half at +0, dO half at +D/64 * 8 KB)
    using C = BCfg<D>;
    constexpr int kItems = C::kStagesKv;        // half-items in the ring
    constexpr uint32_t NB = C::kBufsKv;         // S^T / dP^T buffers
    // d = 64: the warpgroups take alternate half-items (all 64 columns each)
    // instead of sharing each one; with three buffers the chain through a
    // half-item has room for the longer pass, and each pass's fixed costs
    // (tensor-memory round trips, hand-offs) cover twice the columns
    constexpr bool kAlt = D == 64;
    constexpr int kHalfBytes = 64 * D * 2;      // one 64-row bf16 half tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sK = smem;
    uint8_t* sV = smem + C::kTileBytes;
    uint8_t* sR = smem + 2 * C::kTileBytes;  // half-item stage x at x * 2 * kHalfBytes
    __shared__ BShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WlHeader* h = reinterpret_cast<const WlHeader*>(p.wl);
    const BwdHeader* bh = reinterpret_cast<const BwdHeader*>(p.plan);
    int32_t* err_word = const_cast<int32_t*>(&h->error);
    if (h->error != 0) return;
    if (bh->magic != kBwdMagic || bh->hq != p.hq || bh->hkv != p.hkv ||
        bh->q_tokens != p.q_tokens || bh->k_tokens != p.k_tokens || bh->error != 0) {
        if (tid == 0 && blockIdx.x == 0) atomicCAS(err_word, 0, kErrBadWorklist);
        return;
    }
    const WlSlice* slices = reinterpret_cast<const WlSlice*>(p.wl + h->off.slices);
    const BwdUnit* bunits = reinterpret_cast<const BwdUnit*>(p.plan + bh->off_units);
    const int32_t* order = reinterpret_cast<const int32_t*>(p.plan + bh->off_order);
    const int32_t* gsl = reinterpret_cast<const int32_t*>(p.plan + bh->off_gslices);
    const int32_t n = bh->nunits, B = gridDim.x;
    const int32_t G = p.hq / p.hkv;
    // dispatch as the forward worklist says: units claimed at run time in the
    // plan's order (dynamic: cost classes, then group, kv head and key tile),
    // or dealt to the CTAs in snake order of decreasing cost (static)
    const bool dyn = h->dispatch == PVA_DISPATCH_DYNAMIC;
    BwdHeader* bhw = const_cast<BwdHeader*>(bh);
    if (!dyn && (int32_t)blockIdx.x >= n) return;
    // unit readers beyond the MMA and element-wise warps: the loader warp
    if (tid == 0) init_barriers(sh, kItems, 256, 1, 2, 2, kAlt ? 4 : 8);
    // -LSE log2 e and -D of the 64 queries of each staged half-item
    __shared__ __align__(16) float s_nl[kLdSlots][64];
    __shared__ __align__(16) float s_nd[kLdSlots][64];
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmdo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int32_t* abort_flag = &sh.abort_flag;
    // static: units sorted by cost, dealt to the CTAs in snake order: b, 2B-1-b, 2B+b, ...
    auto pos_of = [&](int32_t round) -> int32_t {
        return round * B + ((round & 1) ? B - 1 - (int32_t)blockIdx.x : (int32_t)blockIdx.x);
    };

    // register split (128 * kRegsCtrl + 256 * kRegsElem <= 384 * 168)
    if (kSplitRegs) {
        if (warp < 4) regs_dealloc<kRegsCtrl>();
        else regs_alloc<kRegsElem>();
    }
    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, a_it = 0;
            bool live = true;
            for (uint32_t rd = 0; live; ++rd) {
                live = uring_wait_free(sh.ur, rd, abort_flag, err_word, kErrTimeoutBase + 39,
                                       kWaitNs);
                if (!live) break;
                int32_t pos = dyn ? dispatch_claim(&bhw->dispatch_next) : pos_of((int32_t)rd);
                int32_t idx = pos < n ? order[pos] : -1;
                if (idx >= n || idx < -1) {  // a damaged order: stop, report
                    atomicCAS(err_word, 0, kErrBadWorklist);
                    idx = -1;
                }
                uring_put(sh.ur, rd, idx);
                if (idx < 0) break;
                const BwdUnit u = bunits[idx];
                if (u.cost <= 1) continue;  // no query sees these keys
                const WlSlice s = slices[gsl[u.gbegin]];
                live = mbar_wait(&sh.a_empty, (a_it & 1) ^ 1, abort_flag, err_word,
                                 kErrTimeoutBase + 31, kWaitNs);
                if (!live) break;
                mbar_arrive_expect_tx(&sh.a_full, 2 * C::kTileBytes);
                for (int b = 0; b < D / 64; ++b) {
                    tma_load_3d(sK + b * 16384, &tmk, &sh.a_full, b * 64, u.kvh, s.k_row0 + u.kt * 128);
                    tma_load_3d(sV + b * 16384, &tmv, &sh.a_full, b * 64, u.kvh, s.k_row0 + u.kt * 128);
                }
                ++a_it;
                for (int32_t m = 0; m < u.gcount && live; ++m) {
                    const WlSlice sm = slices[gsl[u.gbegin + m]];
                    int32_t qlo, qhi;
                    bwd_q_span(sm, u.kt, qlo, qhi, slice_mask(p.wl, h, sm, gsl[u.gbegin + m]));
                    for (int32_t t = qlo; t < qhi && live; ++t) {
                        const int32_t nq = min(128, sm.q_len - t * 128);
                        const int32_t halves = nq > 64 ? 2 : 1;
                        for (int32_t hh = 0; hh < G && live; ++hh) {
                            const int32_t head = u.kvh * G + hh;
                            for (int32_t hf = 0; hf < halves && live; ++hf) {
                                const uint32_t st = it % kItems;
                                live = mbar_wait(&sh.r_empty[st], ((it / kItems) & 1) ^ 1,
                                                 abort_flag, err_word, kErrTimeoutBase + 32,
                                                 kWaitNs);
                                if (!live) break;
                                mbar_arrive_expect_tx(&sh.r_full[st], 2 * kHalfBytes);
                                uint8_t* dq_ = sR + st * 2 * kHalfBytes;
                                uint8_t* ddo = dq_ + kHalfBytes;
                                for (int b = 0; b < D / 64; ++b) {
                                    tma_load_3d(dq_ + b * 8192, &tmq, &sh.r_full[st], b * 64, head,
                                                sm.q_row0 + t * 128 + hf * 64);
                                    tma_load_3d(ddo + b * 8192, &tmdo, &sh.r_full[st], b * 64,
                                                head, sm.q_row0 + t * 128 + hf * 64);
                                }
                                ++it;
                            }
                        }
                    }
                }
            }
            if (!live) {
                const uint32_t nn = it < (uint32_t)kItems ? it : (uint32_t)kItems;
                for (uint32_t k = 0; k < nn; ++k) {
                    const uint32_t x = it - 1 - k;
                    mbar_wait_drain(&sh.r_full[x % kItems], (x / kItems) & 1, kDrainNs);
                }
                if (a_it > 0) mbar_wait_drain(&sh.a_full, (a_it - 1) & 1, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------- MMA issuers (whole warps)
        // Half-items: the 64 queries [64 hf, 64 hf + 64) of one (head, slice, q tile)
        // item.  Warp 1 issues S^T = K Q^T and dV += P^T dO, warp 3 dP^T = V dO^T and
        // dK += dS^T Q: one warp spent longer issuing a half-item's 24 MMAs and
        // waiting for its operands than the tensor pipe took to run them.  S^T and
        // dP^T of half-item u go to buffer u % NB (64 columns each); each warp issues
        // them before its dV or dK MMAs of half-item u - NB + 1, so the element-wise
        // warps work on the NB - 1 half-items before u while the tensor pipe computes
        // u.  A warp reuses its half of buffer u % NB only after its own MMAs that
        // read it (issue order); s2_full, r_empty, a_empty and o_full count one commit
        // from each warp.
        const bool sdv = warp == 1;
        const int site = sdv ? 0 : 17;  // wait sites 33-36 (warp 1), 50-53 (warp 3)
        uint32_t it = 0, a_it = 0, gu = 0, o_cnt = 0;
        bool live = true;
        const uint64_t dA = sdesc_sw128(smem_u32(sdv ? sK : sV), 16, 1024);
        const uint64_t dRn = sdesc_sw128(smem_u32(sR), 16, 1024);    // K-major
        const uint64_t dRm = sdesc_sw128(smem_u32(sR), 8192, 1024);  // MN-major, 64-row atoms
        constexpr uint32_t kIdescHalf = idesc_bf16_f32(128, 64, false);
        // this warp's buffer half, accumulator, and the operands of its two GEMMs
        // within a ring stage: S^T reads the Q half, dV the dO half; dP^T the dO
        // half, dK the Q half
        const uint32_t tBuf = tmem + (sdv ? 0 : 64 * NB);
        const uint32_t tAcc = tmem + 128 * NB + (sdv ? 0 : D);
        const uint32_t offN = sdv ? 0 : kHalfBytes, offAcc = sdv ? kHalfBytes : 0;
        // the half-items (oldest first) whose dV or dK MMAs are still to be issued
        bool first = true;
        uint32_t npend = 0, pu0 = 0, pu1 = 0, ps0 = 0, ps1 = 0;  // NB - 1 <= 2 of them
        auto finish_pending = [&]() -> bool {
            const uint32_t pu = pu0, pst = ps0;
            const uint32_t b = pu % NB;
            // the unit's first dV/dK MMAs overwrite the accumulators: the previous
            // unit's epilogue must have read them (waited only here, so that S^T and
            // dP^T of the first half-items overlap that epilogue)
            if (first && !mbar_wait_warp(&sh.o_empty, (o_cnt & 1) ^ 1, abort_flag, err_word,
                                         kErrTimeoutBase + 34 + site, kWaitNs))
                return false;
            if (!mbar_wait_warp(&sh.p2_full[b], (pu / NB) & 1, abort_flag, err_word,
                                kErrTimeoutBase + 36 + site, kWaitNs))
                return false;
            tc_fence_after();
            const uint64_t oB = (pst * 2 * kHalfBytes + offAcc) >> 4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_ts_elect(tAcc, tBuf + 64 * b + kslice_col(k), dRm + oB + k * 128, C::kIdescNN,
                             (!first || k > 0) ? 1u : 0u);
            first = false;
            mma_commit_elect(&sh.r_empty[pst]);
            pu0 = pu1;
            ps0 = ps1;
            --npend;
            return true;
        };
        for (uint32_t rd = 0; live; ++rd) {
            int32_t idx;
            live = uring_get_warp(sh.ur, rd, idx, abort_flag, err_word,
                                  kErrTimeoutBase + (sdv ? 40 : 54), kWaitNs);
            if (!live || idx < 0) break;
            const BwdUnit u = bunits[idx];
            if (u.cost <= 1) continue;
            live = mbar_wait_warp(&sh.a_full, a_it & 1, abort_flag, err_word,
                                  kErrTimeoutBase + 33 + site, kWaitNs);
            if (!live) break;
            first = true;
            for (int32_t m = 0; m < u.gcount && live; ++m) {
                const WlSlice sm = slices[gsl[u.gbegin + m]];
                int32_t qlo, qhi;
                bwd_q_span(sm, u.kt, qlo, qhi, slice_mask(p.wl, h, sm, gsl[u.gbegin + m]));
                for (int32_t t = qlo; t < qhi && live; ++t) {
                    const int32_t nq = min(128, sm.q_len - t * 128);
                    const uint32_t halves = nq > 64 ? 2 : 1;
                    for (int32_t hh = 0; hh < G && live; ++hh) {
                        for (uint32_t hf = 0; hf < halves && live; ++hf) {
                            const uint32_t st = it % kItems;
                            live = mbar_wait_warp(&sh.r_full[st], (it / kItems) & 1, abort_flag,
                                                  err_word, kErrTimeoutBase + 35 + site, kWaitNs);
                            if (!live) break;
                            tc_fence_after();
                            const uint32_t b = gu % NB;
                            const uint64_t oN = (st * 2 * kHalfBytes + offN) >> 4;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                // K or V (resident, 128-row atoms) against the Q or dO
                                // half (64-row atoms)
                                const uint32_t kq = (k >> 2) * 512 + (k & 3) * 2;
                                const uint32_t off16 = (k >> 2) * 1024 + (k & 3) * 2;
                                mma_ss_elect(tBuf + 64 * b, dA + off16, dRn + oN + kq, kIdescHalf,
                                             k > 0);
                            }
                            mma_commit_elect(&sh.s2_full[b]);
                            if (npend == NB - 1 && !finish_pending()) {
                                live = false;
                                break;
                            }
                            if (npend == 0) {
                                pu0 = gu;
                                ps0 = st;
                            } else {
                                pu1 = gu;
                                ps1 = st;
                            }
                            ++npend;
                            ++gu;
                            ++it;
                        }
                    }
                }
            }
            if (!live) break;
            while (npend > 0 && finish_pending()) {
            }
            if (npend > 0) break;
            mma_commit_elect(&sh.a_empty);
            mma_commit_elect(&sh.o_full);
            ++o_cnt;
            ++a_it;
        }
        uint64_t* done = sdv ? &sh.done : &sh.done2;
        mma_commit_elect(done);
        mbar_wait_drain(done, 0, kDrainNs);
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------- (LSE, D) loader
        // Walks the half-items in the element-wise warps' order and stages -LSE
        // log2 e and -D of their 64 queries up to kLdSlots half-items ahead, so
        // the global-load latency stays off the element-wise warps' path.  A
        // query past the tile gets LSE = +inf: every P of it is 0.
        uint32_t li = 0;
        bool live = true;
        for (uint32_t rd = 0; live; ++rd) {
            int32_t idx;
            live = uring_get_warp(sh.ur, rd, idx, abort_flag, err_word, kErrTimeoutBase + 41,
                                  kWaitNs);
            if (!live || idx < 0) break;
            const BwdUnit u = bunits[idx];
            if (u.cost <= 1) continue;
            for (int32_t m = 0; m < u.gcount && live; ++m) {
                const WlSlice s = slices[gsl[u.gbegin + m]];
                int32_t qlo, qhi;
                bwd_q_span(s, u.kt, qlo, qhi, slice_mask(p.wl, h, s, gsl[u.gbegin + m]));
                for (int32_t t = qlo; t < qhi && live; ++t) {
                    const int32_t qrow0 = s.q_row0 + t * 128;
                    const int32_t nq = min(128, s.q_len - t * 128);
                    const uint32_t halves = nq > 64 ? 2 : 1;
                    for (int32_t hh = 0; hh < G && live; ++hh) {
                        const int32_t head = u.kvh * G + hh;
                        for (uint32_t hf = 0; hf < halves && live; ++hf, ++li) {
                            const uint32_t slot = li % kLdSlots;
                            live = mbar_wait_warp(&sh.ld_empty[slot], ((li / kLdSlots) & 1) ^ 1,
                                                  abort_flag, err_word, kErrTimeoutBase + 42,
                                                  kWaitNs);
                            if (!live) break;
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                const int qc = (int)hf * 64 + c * 32 + lane;
                                float l2 = INFINITY, dd = 0.f;
                                if (qc < nq) {
                                    const int64_t li_ = (int64_t)head * p.q_tokens + qrow0 + qc;
                                    const float l = p.lse[li_];
                                    if (l != -INFINITY) l2 = l * 1.4426950408889634f;
                                    dd = p.dvec[li_];
                                }
                                s_nl[slot][c * 32 + lane] = -l2;
                                s_nd[slot][c * 32 + lane] = -dd;
                            }
                            mbar_arrive(&sh.ld_full[slot]);  // every lane, after its writes
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------- P^T, dS^T and the dK/dV epilogue
        // d = 128: two warpgroups share every half-item, wg taking its 32 query
        // columns [32 wg, 32 wg + 32), so a half-item's P^T and dS^T are ready in
        // half the time; d = 64: warpgroup u % 2 takes half-item u.  At the end
        // of a unit wg 0 stores dV and wg 1 dK.
        const int wg = (warp - 4) >> 2;
        const int kr = (warp & 3) * 32 + lane;  // key row = tensor-memory lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base, tV = tmem + lane_base + 128 * NB,
                       tK = tmem + lane_base + 128 * NB + D;
        uint32_t gu = 0, o_cnt = 0, li = 0;
        bool live = true;
        for (uint32_t rd = 0; live; ++rd) {
            int32_t idx;
            live = uring_get(sh.ur, rd, idx, abort_flag, err_word, kErrTimeoutBase + 40, kWaitNs);
            if (!live || idx < 0) break;
            const BwdUnit u = bunits[idx];
            const WlSlice s0 = slices[gsl[u.gbegin]];  // the group's key range
            const int32_t krows = min(128, s0.k_len - u.kt * 128);
            const bool kvalid = kr < krows;
            const int64_t grow = ((int64_t)(s0.k_row0 + u.kt * 128 + kr) * p.hkv + u.kvh) * D;
            if (u.cost <= 1) {  // keys no query sees: zero gradient
                if (kvalid) {
                    store_zero_row(wg == 0 ? p.dv : p.dk, grow, p.grads_fp32, D);
                }
                continue;
            }
            for (int32_t m = 0; m < u.gcount && live; ++m) {
                const WlSlice s = slices[gsl[u.gbegin + m]];
                const uint32_t* pm = slice_mask(p.wl, h, s, gsl[u.gbegin + m]);
                const int32_t k_pos = s.k_pos0 + u.kt * 128 + kr;
                int64_t qa, qb;  // query positions that may see this key
                slice_queries_of_key(s, k_pos, qa, qb, pm);
                int32_t qlo, qhi;
                bwd_q_span(s, u.kt, qlo, qhi, pm);
                for (int32_t t = qlo; t < qhi && live; ++t) {
                    // this q tile's rows: query c has position q_pos0 + t*128 + c
                    const int32_t nq = min(128, s.q_len - t * 128);
                    const int32_t cpos0 = s.q_pos0 + t * 128;
                    const int32_t c_lo = (int32_t)max((int64_t)0, qa - cpos0);
                    const int32_t c_hi = kvalid ? (int32_t)min((int64_t)nq, qb - cpos0) : 0;
                    const uint32_t halves = nq > 64 ? 2 : 1;
                    for (int32_t hh = 0; hh < G && live; ++hh) {
                    for (uint32_t hf = 0; hf < halves && live; ++hf, ++gu) {
                        const uint32_t b = gu % NB;
                        if (kAlt && (gu & 1) != (uint32_t)wg) {  // the other warpgroup's
                            ++li;
                            continue;
                        }
                        // the staged -LSE log2 e and -D of the half's 64 queries; a query
                        // past the tile has LSE = +inf, so every P of it is 0
                        const uint32_t slot = li % kLdSlots;
                        live = mbar_wait(&sh.ld_full[slot], (li / kLdSlots) & 1, abort_flag,
                                         err_word, kErrTimeoutBase + 43, kWaitNs);
                        if (!live) break;
                        // columns [c_lo, c_hi) of this key row are allowed; the warp masks a
                        // chunk of 32 only when some row of it has a limit inside the chunk
                        // (d = 128: decided before the wait for S^T; d = 64 per chunk, which
                        // needs fewer registers)
                        const int hw = (int)hf * 64 + wg * 32;
                        const bool mask_w =
                            !kAlt && __any_sync(0xffffffffu, c_lo > hw || c_hi < min(hw + 32, nq));
                        live = mbar_wait(&sh.s2_full[b], (gu / NB) & 1, abort_flag, err_word,
                                         kErrTimeoutBase + 37, kWaitNs);
                        if (!live) break;
                        tc_fence_after();
                        const uint32_t tSb = tS + 64 * b, tPb = tS + 64 * NB + 64 * b;
                        // P^T and dS^T of query columns [h0, h0 + 32) of the q tile, packed
                        // over the first 16 of the chunk's S^T and dP^T columns
                        auto chunk = [&](const int c, const bool need_mask) {
                            const int h0 = (int)hf * 64 + c * 32;
                            const float* my_nl = s_nl[slot] + c * 32;
                            const float* my_nd = s_nd[slot] + c * 32;
                            uint32_t sv[32], pv[32];
                            tmem_ld32(tSb + c * 32, sv);
                            tmem_ld32(tPb + c * 32, pv);
                            tmem_ld_wait(sv);
                            tmem_ld_wait(pv);
                            uint32_t pw[32], dw[32];
                            const float2 sc = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                const float4 nl = *reinterpret_cast<const float4*>(&my_nl[e]);
                                const float4 nd = *reinterpret_cast<const float4*>(&my_nd[e]);
#pragma unroll
                                for (int j = 0; j < 4; j += 2) {
                                    const float2 x = __ffma2_rn(
                                        make_float2(__uint_as_float(sv[e + j]),
                                                    __uint_as_float(sv[e + j + 1])),
                                        sc, j == 0 ? make_float2(nl.x, nl.y)
                                                   : make_float2(nl.z, nl.w));
                                    float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
                                    if (need_mask) {
                                        const int col = h0 + e + j;
                                        if (col < c_lo || col >= c_hi) p0 = 0.f;
                                        if (col + 1 < c_lo || col + 1 >= c_hi) p1 = 0.f;
                                    }
                                    const float2 g = __fmul2_rn(
                                        make_float2(p0, p1),
                                        __fadd2_rn(make_float2(__uint_as_float(pv[e + j]),
                                                               __uint_as_float(pv[e + j + 1])),
                                                   j == 0 ? make_float2(nd.x, nd.y)
                                                          : make_float2(nd.z, nd.w)));
                                    pw[(e + j) >> 1] = pack_bf16x2(p0, p1);
                                    dw[(e + j) >> 1] = pack_bf16x2(g.x, g.y);
                                }
                            }
                            tmem_st16(tSb + c * 32, pw);
                            tmem_st16(tPb + c * 32, dw);
                        };
                        if constexpr (kAlt) {
#pragma unroll 1
                            for (int c = 0; c < 2; ++c) {
                                const int h0 = (int)hf * 64 + c * 32;
                                chunk(c, __any_sync(0xffffffffu,
                                                    c_lo > h0 || c_hi < min(h0 + 32, nq)));
                            }
                        } else {
                            chunk(wg, mask_w);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();  // also: every lane has read its staged (LSE, D)
                        if (lane == 0) {
                            mbar_arrive(&sh.p2_full[b]);
                            mbar_arrive(&sh.ld_empty[slot]);
                        }
                        ++li;
                    }
                    }
                }
            }
            if (!live) break;
            live = mbar_wait(&sh.o_full, o_cnt & 1, abort_flag, err_word, kErrTimeoutBase + 38,
                             kWaitNs);
            if (!live) break;
            ++o_cnt;
            tc_fence_after();
            // wg 0: dV = P^T dO; wg 1: dK = scale dS^T Q
            const uint32_t tOut = wg == 0 ? tV : tK;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t a[32];
                tmem_ld32(tOut + c * 32, a);
                tmem_ld_wait(a);
                if (kvalid)
                    store_row32(wg == 0 ? p.dv : p.dk, grow + c * 32, p.grads_fp32, a,
                                wg == 0 ? 1.f : p.scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.o_empty);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (dyn && tid == 0) dispatch_exit(&bhw->dispatch_next, &bhw->dispatch_done);
}

template <int D>
pva_status launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const CUtensorMap& mdo, const CUtensorMap& mq64, const CUtensorMap& mdo64,
                      const CUtensorMap& mk64, const CUtensorMap& mv64, const BwdParams& bp,
                      int32_t dkdv_ctas, cudaStream_t st) {
    const int grid_pre = 4 * bp.num_ctas;
    bwd_pre_kernel<<<grid_pre, 256, 0, st>>>(bp);
    auto kq = bwd_dq_kernel<D>;
    auto kk = bwd_dkdv_kernel<D>;
    // setmaxnreg.inc draws from the registers the block was launched with: the
    // dK/dV split must fit in (threads x registers per thread)
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kk) != cudaSuccess) return PVA_ERR_CUDA;
    if (kSplitRegs &&
        (int64_t)fa.numRegs * kThreads < 128 * (int64_t)kRegsCtrl + 256 * (int64_t)kRegsElem)
        return PVA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<D>::kSmemDq) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<D>::kSmemKv) !=
            cudaSuccess)
        return PVA_ERR_CUDA;
    kq<<<bp.num_ctas, kThreads, BCfg<D>::kSmemDq, st>>>(mq, mk64, mv64, mdo, bp);
    kk<<<dkdv_ctas, kThreads, BCfg<D>::kSmemKv, st>>>(mq64, mk, mv, mdo64, bp);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pva

using namespace pva;

extern "C" pva_status pva_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                                   const float* lse, const void* dout,
                                   const int32_t* cu_seqlens_dev, int32_t num_docs,
                                   const pva_mask_desc* mask,
                                   const pva_worklist_params* params, int32_t head_dim,
                                   const void* worklist_dev, void* plan_dev, void* dq, void* dk,
                                   void* dv, int32_t grads_are_fp32, float softmax_scale,
                                   void* stream) {
    if (!mask || !params || !worklist_dev || !plan_dev || !q || !out || !lse || !dout || !dq ||
        !dk || !dv)
        return PVA_ERR_INVALID_ARG;
    if (mask->kind != PVA_MASK_SLICES && !cu_seqlens_dev) return PVA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PVA_ERR_UNSUPPORTED;
    if (params->tile_m != 128 || params->tile_n != 128) return PVA_ERR_UNSUPPORTED;
    if (params->num_q_heads <= 0 || params->num_kv_heads <= 0 ||
        params->num_q_heads % params->num_kv_heads != 0)
        return PVA_ERR_INVALID_ARG;
    if (grads_are_fp32 != 0 && grads_are_fp32 != 1) return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens < 0 || mask->k_tokens < 0) return PVA_ERR_INVALID_ARG;
    if (mask->k_tokens > 0 && (!k || !v)) return PVA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(dout) || !aligned16(lse) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) ||
        (mask->k_tokens > 0 && (!aligned16(k) || !aligned16(v))) ||
        (reinterpret_cast<uintptr_t>(worklist_dev) & 255u) ||
        (reinterpret_cast<uintptr_t>(plan_dev) & 255u))
        return PVA_ERR_INVALID_ARG;
    const int32_t nc = resolve_num_ctas(params->num_ctas);
    if (nc <= 0) return PVA_ERR_CUDA;
    if (nc > kMaxBins) return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = grads_are_fp32 ? 4 : 2;
    // Keys that no slice covers get no gradient: explicit slices, and a zigzag
    // pair's (or ring step's) key chunks that lie after every query chunk of
    // their document.
    // Queries outside every segment: explicit slices only.
    if (mask->kind == PVA_MASK_SLICES &&
        cudaMemsetAsync(dq, 0, (size_t)mask->q_tokens * params->num_q_heads * head_dim * es, st) !=
            cudaSuccess)
        return PVA_ERR_CUDA;
    if ((mask->kind == PVA_MASK_SLICES || mask->kind == PVA_MASK_ZIGZAG_PAIR ||
         mask->kind == PVA_MASK_ZIGZAG_STEP) &&
        (cudaMemsetAsync(dk, 0, (size_t)mask->k_tokens * params->num_kv_heads * head_dim * es,
                         st) != cudaSuccess ||
         cudaMemsetAsync(dv, 0, (size_t)mask->k_tokens * params->num_kv_heads * head_dim * es,
                         st) != cudaSuccess))
        return PVA_ERR_CUDA;
    if (mask->q_tokens == 0) return PVA_OK;
    // the plan's D scratch (its header is checked on the device)
    const int64_t off_dvec = bwd_plan_dvec_offset(num_docs, mask, params);
    if (off_dvec < 0) return PVA_ERR_INVALID_ARG;
    CUtensorMap mq, mk, mv, mdo, mq64, mdo64, mk64, mv64;
    const void* kp = mask->k_tokens > 0 ? k : q;
    const void* vp = mask->k_tokens > 0 ? v : q;
    const int32_t kh = mask->k_tokens > 0 ? params->num_kv_heads : params->num_q_heads;
    if (!make_map(&mq, q, mask->q_tokens, params->num_q_heads, head_dim) ||
        !make_map(&mk, kp, mask->k_tokens, kh, head_dim) ||
        !make_map(&mv, vp, mask->k_tokens, kh, head_dim) ||
        !make_map(&mdo, dout, mask->q_tokens, params->num_q_heads, head_dim) ||
        !make_map(&mq64, q, mask->q_tokens, params->num_q_heads, head_dim, 64) ||
        !make_map(&mdo64, dout, mask->q_tokens, params->num_q_heads, head_dim, 64) ||
        !make_map(&mk64, kp, mask->k_tokens, kh, head_dim, 64) ||
        !make_map(&mv64, vp, mask->k_tokens, kh, head_dim, 64))
        return PVA_ERR_CUDA;
    BwdParams bp;
    bp.wl = reinterpret_cast<const uint8_t*>(worklist_dev);
    bp.plan = reinterpret_cast<const uint8_t*>(plan_dev);
    bp.out = out;
    bp.dout = dout;
    bp.lse = lse;
    bp.dvec = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(plan_dev) + off_dvec);
    bp.dq = dq;
    bp.dk = dk;
    bp.dv = dv;
    bp.q_tokens = mask->q_tokens;
    bp.k_tokens = mask->k_tokens;
    bp.hq = params->num_q_heads;
    bp.hkv = params->num_kv_heads;
    bp.grads_fp32 = grads_are_fp32;
    bp.num_ctas = nc;
    bp.d = head_dim;
    bp.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
    bp.scale_log2 = bp.scale * 1.4426950408889634f;
    return head_dim == 128 ? launch_bwd<128>(mq, mk, mv, mdo, mq64, mdo64, mk64, mv64, bp, nc, st)
                           : launch_bwd<64>(mq, mk, mv, mdo, mq64, mdo64, mk64, mv64, bp, nc, st);
}
