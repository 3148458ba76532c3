// attn_fwd.cu -- persistent packed document-masked attention forward on
// sm_103a (tcgen05 MMAs into tensor memory, TMA-staged tiles).
//
// The method: "03 · 长文负载均衡" §1.1 (each document attends only to itself;
// the quadratic work is QK^T and PV), §3.2 (only (Q block, KV block) pairs
// with a non-zero mask are computed; partial results over key blocks are
// combined by online-softmax rescale-and-sum), §1.2 (structured masks).
//
// One CTA per SM runs work units until none is left: under dynamic dispatch
// it claims the next unit of the worklist's dispatch order from a counter
// (LPT rule, "数据并行负载均衡" §4.4, decided by measured time), under static
// dispatch it walks its LPT-assigned list.  A unit holds up to two 128-row
// query sub-tiles that share one kv head and the same kv tiles.  Warp roles
// (384 threads, 3 warpgroups):
//   warp 0      TMA producer: picks the units (unit_feed.cuh ring), loads the
//               Q sub-tiles, then the K / V tiles into a ring
//   warps 1, 2  MMA issuers, one per sub-tile (one elected lane issues):
//               S_i = Q_i K_j^T (SS), O_i += P_i V_j (TS: P read from tensor
//               memory), completion via tcgen05.commit
//   warps 4-7   softmax + epilogue of sub-tile 0 (one query row per thread)
//   warps 8-11  softmax + epilogue of sub-tile 1
// A warp reaches tensor-memory lanes 32*(warp % 4).
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,..),
// O1 [384,..).  At d = 128 P (bf16) overwrites the first half of S in place,
// so QK of tile j+1 follows PV of tile j; at d = 64 P has its own 64 columns
// after O (Cfg::kSplitP) and QK of tile j+1 runs as soon as the softmax has
// read S_j.  With the 32x32b tensor-memory layout a thread owns a whole row,
// so the row max and row sum of the online softmax are thread-local.
// The running max is only moved (and O rescaled in tensor memory) when it
// grows by more than 2^8 in the base-2 exponent domain; until then P stays
// below 2^8, which fp32 and bf16 hold exactly enough.
//
// Every wait is bounded; on timeout the CTA raises an abort flag, records
// the wait site in the worklist error word, drains its own copies and MMAs,
// frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pva.h"
#include "common.h"
#include "ptx.cuh"
#include "tma_map.h"
#include "unit_feed.cuh"
#include "wl_layout.cuh"

namespace pva {
namespace {

constexpr int kThreads = 384;
// register split: the producer/MMA warpgroup hands registers to the two
// softmax warpgroups (128 * ctrl + 256 * softmax <= 384 * 168; multiples of 8):
// 72 / 216 at d = 128, 56 / 224 at d = 64 (fewer softmax spills there)
template <int D>
struct Regs {
    static constexpr uint32_t kCtrl = D == 64 ? 56 : 72, kSoftmax = D == 64 ? 224 : 216;
};
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait
constexpr float kRescaleThreshold = 8.0f;     // log2 domain
constexpr int kURing = 8;                     // units the producer may run ahead
// readers of a unit slot: the two MMA warps (one arrival each) and every
// softmax thread
constexpr uint32_t kUReaders = 2 + 256;

template <int D>
struct Cfg {
    static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
    static constexpr int kStages = D == 128 ? 4 : 8;
    // d = 64 leaves 64 free tensor-memory columns per sub-tile: P goes there
    // instead of over S, so QK of the next kv tile need not wait for PV
    static constexpr bool kSplitP = D == 64;
    // K/V ring: one tile per stage; with kSplitP a stage holds K_{j+1} (at +0) and
    // V_j (at +kTileBytes), waited for and released once per kv tile
    static constexpr int kRingStages = kSplitP ? kStages / 2 : kStages;
    static constexpr int kStageBytes = kSplitP ? 2 * kTileBytes : kTileBytes;
    // per softmax warp, 32 rows x 128 bytes of O staged for a TMA store
    static constexpr int kStageOutBytes = 8 * 4096;
    static constexpr int kSmem = 2 * kTileBytes + kStages * kTileBytes + kStageOutBytes + 1024;
    static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, true);
};

struct AttnParams {
    const uint8_t* wl;
    void* out;
    float* lse;
    uint64_t* busy;
    int32_t q_tokens, k_tokens, hq, hkv, out_fp32, num_ctas;
    float scale_log2;
    int32_t accumulate;   // merge into the running fp32 (out, lse) instead of writing
                          // (selects the kernel instantiation)
    int32_t withhold_kv;  // test hook: the producer of CTA 0 (static dispatch) or of the CTA
                          // that claimed LPT rank 0 (dynamic) skips its K/V item 1
    int32_t dynamic;      // 1: claim units in LPT order from the worklist's counter
};

struct SubTile {
    int32_t q_row, nrows, q_pos, head;
};

struct Unit {
    int32_t nsub, kvh, run_begin, run_count, ntiles;
    SubTile st[2];
};

__device__ __forceinline__ Unit decode_unit(const WlUnit& u, const WlSeg* segs) {
    const WlSeg g = segs[u.seg];
    Unit r;
    r.nsub = u.h1 >= 0 ? 2 : 1;
    r.kvh = u.kvh;
    r.run_begin = u.run_begin;
    r.run_count = u.run_count;
    r.ntiles = u.ntiles;
    const int32_t ts[2] = {u.t0, u.t1};
    const int32_t hs[2] = {u.h0, u.h1};
    for (int i = 0; i < 2; ++i) {
        const int32_t t = ts[i] >= 0 ? ts[i] : 0;
        r.st[i].q_row = g.q_row0 + t * 128;
        r.st[i].nrows = min(128, g.q_len - t * 128);
        r.st[i].q_pos = g.q_pos0 + t * 128;
        r.st[i].head = hs[i];
    }
    return r;
}

struct Shared {
    uint64_t q_full[2], q_empty[2], s_full[2], p_half[2], p_full[2], o_full[2], o_empty[2], done[2],
        turn[2];
    // C::kSplitP only: S read by the softmax (4 warp arrivals), PV complete (commit)
    uint64_t s_free[2], pv_done[2];
    uint64_t kv_full[8], kv_empty[8];
    UnitRing<kURing> ur;  // the producer hands each unit's index to the other roles
    uint32_t tmem_base;
    int32_t abort_flag;
};

__device__ __forceinline__ void write_empty_rows(const AttnParams& p, const SubTile& st, int r,
                                                 int D) {
    if (r >= st.nrows) return;
    const int64_t row = (int64_t)(st.q_row + r) * p.hq + st.head;
    if (p.out_fp32) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * D);
        for (int c = 0; c < D / 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * D);
        for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
    }
    p.lse[(int64_t)st.head * p.q_tokens + st.q_row + r] = -INFINITY;
}

// ACC: the fused ring step (pva_attn_fwd_accumulate), a separate instantiation
// so that each kernel carries only the epilogue it runs.
template <int D, bool ACC>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                    const AttnParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ[2] = {smem, smem + C::kTileBytes};
    uint8_t* sKV = smem + 2 * C::kTileBytes;
    uint8_t* sStage = sKV + C::kStages * C::kTileBytes;  // 4 KB per softmax warp, 1 KB aligned
    __shared__ Shared sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WlHeader* h = reinterpret_cast<const WlHeader*>(p.wl);
    int32_t* err_word = const_cast<int32_t*>(&h->error);
    // the worklist must describe this call
    const bool ok = h->magic == kWlMagic && h->tile_m == 128 && h->tile_n == 128 &&
                    h->hq == p.hq && h->hkv == p.hkv && h->num_ctas == p.num_ctas &&
                    (int)gridDim.x == p.num_ctas && h->q_tokens == p.q_tokens &&
                    h->k_tokens == p.k_tokens &&
                    (h->dispatch == PVA_DISPATCH_DYNAMIC) == (p.dynamic != 0);
    if (!ok) {
        if (tid == 0 && blockIdx.x == 0) atomicCAS(err_word, 0, kErrBadWorklist);
        return;
    }
    if (h->error != 0) return;  // the build failed: nothing is written
    const int32_t* cta_off = reinterpret_cast<const int32_t*>(p.wl + h->off.cta_off);
    const WlUnit* units = reinterpret_cast<const WlUnit*>(p.wl + h->off.units);
    const WlRun* runs = reinterpret_cast<const WlRun*>(p.wl + h->off.runs);
    const WlSlice* slices = reinterpret_cast<const WlSlice*>(p.wl + h->off.slices);
    const WlSeg* segs = reinterpret_cast<const WlSeg*>(p.wl + h->off.segs);
    // Static dispatch: this CTA's CSR list of `units`.  Dynamic dispatch: the
    // CTA claims ranks one by one from the worklist's counter and runs
    // units_enum[dorder[rank]], so a unit goes to whichever CTA frees up first
    // (list scheduling over power-of-two cost classes in decreasing order;
    // inside a class, enumeration order keeps concurrent units on the same
    // documents' K/V in L2).
    const int32_t* order = reinterpret_cast<const int32_t*>(p.wl + h->off.dorder);
    const WlUnit* ubase =
        p.dynamic ? reinterpret_cast<const WlUnit*>(p.wl + h->off.units_enum) : units;
    WlHeader* hw = const_cast<WlHeader*>(h);
    const int32_t nunits = h->nunits;
    // (a dynamic-dispatch worklist has no per-CTA lists)
    const int32_t ub = p.dynamic ? 0 : cta_off[blockIdx.x];
    const int32_t ue = p.dynamic ? 0 : cta_off[blockIdx.x + 1];
    const uint64_t t_start = globaltimer_ns();
    if (!p.dynamic && ub >= ue) {
        if (p.busy && tid == 0) {
            p.busy[2 * blockIdx.x] = t_start;
            p.busy[2 * blockIdx.x + 1] = t_start;
        }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.q_full[i], 1);
            mbar_init(&sh.q_empty[i], 1);
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_half[i], 4);   // one arrival per softmax warp
            mbar_init(&sh.p_full[i], 4);
            mbar_init(&sh.o_full[i], 1);
            mbar_init(&sh.o_empty[i], 128);
            mbar_init(&sh.done[i], 1);
            mbar_init(&sh.turn[i], 1);
            mbar_init(&sh.s_free[i], 4);
            mbar_init(&sh.pv_done[i], 1);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&sh.kv_full[s], 1);
            mbar_init(&sh.kv_empty[s], 2);
        }
        uring_init(sh.ur, kUReaders);
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int32_t* abort_flag = &sh.abort_flag;

    // every role ends here: all 384 threads meet, warp 1 frees tensor memory
    auto finish = [&]() {
        // the output stores issued from the staging buffers have completed
        if (warp >= 4 && lane == 0) bulk_wait_all();
        tc_fence_before();
        named_barrier(1, kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        if (p.busy && tid == 0) {
            p.busy[2 * blockIdx.x] = t_start;
            p.busy[2 * blockIdx.x + 1] = globaltimer_ns();
        }
        // every claim of this CTA came before its finish; the last CTA to
        // finish leaves the counter at 0 for the next launch on this worklist
        if (p.dynamic && tid == 0) dispatch_exit(&hw->dispatch_next, &hw->dispatch_done);
    };
    if (warp < 4) {
      regs_dealloc<Regs<D>::kCtrl>();
      if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t kv_it = 0, q_it[2] = {0, 0};
            bool live = true;
            bool hook = p.withhold_kv && !p.dynamic && blockIdx.x == 0;
            for (uint32_t nu = 0; live; ++nu) {
                live = uring_wait_free(sh.ur, nu, abort_flag, err_word, kErrTimeoutBase + 13,
                                       kWaitNs);
                if (!live) break;
                int32_t idx;
                if (p.dynamic) {
                    // claimed once this CTA's producer has issued every load of
                    // its previous unit, a few K/V steps before the CTA needs it
                    const int32_t rank = dispatch_claim(&hw->dispatch_next);
                    idx = rank < nunits ? order[rank] : -1;
                    if (idx >= nunits || idx < -1) {  // a damaged order: stop, report
                        atomicCAS(err_word, 0, kErrBadWorklist);
                        idx = -1;
                    }
                    if (rank == 0 && p.withhold_kv) hook = true;
                } else {
                    idx = ub + (int32_t)nu < ue ? ub + (int32_t)nu : -1;
                }
                uring_put(sh.ur, nu, idx);
                if (idx < 0) break;
                const WlUnit wu = ubase[idx];
                const Unit u = decode_unit(wu, segs);
                if (u.ntiles == 0) continue;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i >= u.nsub || !live) break;
                    live = mbar_wait(&sh.q_empty[i], (q_it[i] & 1) ^ 1, abort_flag, err_word,
                                     kErrTimeoutBase + 1, kWaitNs);
                    if (!live) break;
                    mbar_arrive_expect_tx(&sh.q_full[i], C::kTileBytes);
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(sQ[i] + b * 16384, &tmq, &sh.q_full[i], b * 64, u.st[i].head,
                                    u.st[i].q_row);
                    ++q_it[i];
                }
                // the next ring stage: the K tile of key row krow_k and/or the V tile of
                // krow_v (-1: none)
                auto load_stage = [&](int32_t krow_k, int32_t krow_v) {
                    if (hook && kv_it == 1) {
                        ++kv_it;  // test hook: this copy never arrives
                        return;
                    }
                    const uint32_t st = kv_it % C::kRingStages;
                    live = mbar_wait(&sh.kv_empty[st], ((kv_it / C::kRingStages) & 1) ^ 1,
                                     abort_flag, err_word, kErrTimeoutBase + 2, kWaitNs);
                    if (!live) return;
                    const uint32_t bytes =
                        (uint32_t)((krow_k >= 0 ? 1 : 0) + (krow_v >= 0 ? 1 : 0)) * C::kTileBytes;
                    mbar_arrive_expect_tx(&sh.kv_full[st], bytes);
                    uint8_t* dst = sKV + st * C::kStageBytes;
                    if (krow_k >= 0)
                        for (int b = 0; b < D / 64; ++b)
                            tma_load_3d(dst + b * 16384, &tmk, &sh.kv_full[st], b * 64, u.kvh,
                                        krow_k);
                    if (krow_v >= 0)
                        for (int b = 0; b < D / 64; ++b)
                            tma_load_3d(dst + (C::kSplitP ? C::kTileBytes : 0) + b * 16384, &tmv,
                                        &sh.kv_full[st], b * 64, u.kvh, krow_v);
                    ++kv_it;
                };
                // the MMA warps' order: K_j, V_j per tile; with kSplitP the stages
                // (K_0), (K_1, V_0), (K_2, V_1), ..., (V_{n-1})
                int32_t pend_v = -1;
                for (int32_t r = 0; r < u.run_count && live; ++r) {
                    const WlRun run = runs[u.run_begin + r];
                    const WlSlice s = slices[run.slice];
                    for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                        const int32_t krow = s.k_row0 + jt * 128;
                        if (C::kSplitP) {
                            load_stage(krow, pend_v);
                            pend_v = krow;
                        } else {
                            load_stage(krow, -1);
                            if (!live) break;
                            load_stage(-1, krow);
                        }
                    }
                }
                if (C::kSplitP && live && pend_v >= 0) load_stage(-1, pend_v);
            }
            if (!live) {
                // drain: wait for the copies this thread issued last
                const uint32_t n =
                    kv_it < (uint32_t)C::kRingStages ? kv_it : (uint32_t)C::kRingStages;
                for (uint32_t k = 0; k < n; ++k) {
                    const uint32_t it = kv_it - 1 - k;
                    mbar_wait_drain(&sh.kv_full[it % C::kRingStages], (it / C::kRingStages) & 1,
                                    kDrainNs);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (q_it[i] > 0) mbar_wait_drain(&sh.q_full[i], (q_it[i] - 1) & 1, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------- MMA issuers
        // Warp 1 issues sub-tile 0's MMAs and warp 2 sub-tile 1's.  An MMA
        // instruction waits for room in the tensor pipe's short queue, so a
        // single issuing thread would reach the second sub-tile's waits only
        // after the first sub-tile's group had nearly drained; with one
        // issuer per sub-tile the next group is queued the moment it may go.
        // In units with two sub-tiles the groups still alternate (QK_0, QK_1,
        // then PV_0 + QK_0, PV_1 + QK_1 per K/V tile) through a turn token, so
        // that the two softmax warpgroups stay half a step apart.
        // Both issuers walk every K/V item in ring order; a stage is free once
        // both have released it (kv_empty counts 2 arrivals).
        const int i = warp - 1;
        // the whole warp runs the loop; one elected lane issues each operation
        {
            uint32_t kv_it = 0, q_it = 0, p_cnt = 0, o_cnt = 0, g = 0;
            bool live = true;
            // group g of this issuer goes after group g - 1 (i = 0) or g (i = 1)
            // of the other one
            auto take_turn = [&](bool pair) -> bool {
                if (!pair) return true;
                if (i == 0 && g == 0) return true;
                return mbar_wait_warp(&sh.turn[i], (i == 0 ? g - 1 : g) & 1, abort_flag, err_word,
                                 kErrTimeoutBase + 11, kWaitNs);
            };
            auto pass_turn = [&](bool pair) {
                if (!pair) return;
                mbar_arrive_elect(&sh.turn[i ^ 1]);
                ++g;
            };
            // Descriptors are built once; an MMA only adds a byte offset >> 4 to the
            // 14-bit start-address field (shared addresses stay below 256 KB).
            const uint64_t dQ = sdesc_sw128(smem_u32(sQ[i]), 16, 1024);
            const uint64_t dK0 = sdesc_sw128(smem_u32(sKV), 16, 1024);     // K-major
            const uint64_t dV0 = sdesc_sw128(smem_u32(sKV), 16384, 1024);  // MN-major
            const uint32_t tS = tmem + i * 128, tO = tmem + 256 + i * 128;
            // a sub-tile this unit lacks still frees each stage after its load landed
            auto release = [&](bool mine, uint32_t st) {
                if (mine) mma_commit_elect(&sh.kv_empty[st]);
                else mbar_arrive_elect(&sh.kv_empty[st]);
            };
            if constexpr (C::kSplitP) {
            // P in its own columns (tP): QK of kv tile j+1 is issued as soon as the
            // softmax has read S_j (s_free), before PV of tile j; the two issuers
            // run independently.  Ring stages: (K_0), then (K_{j+1}, V_j) per tile.
            const uint32_t tP = tO + 64;
            uint32_t s_used = 0;  // QKs issued into S_i
            auto issue_qk = [&](uint32_t st) {
                // S_i is free once the softmax has read the previous S
                if (s_used > 0)
                    live = mbar_wait_warp(&sh.s_free[i], (s_used - 1) & 1, abort_flag, err_word,
                                          kErrTimeoutBase + 15, kWaitNs);
                if (!live) return;
                tc_fence_after();
                const uint64_t dK = dK0 + ((st * C::kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off16 = (k >> 2) * 1024 + (k & 3) * 2;
                    mma_ss_elect(tS, dQ + off16, dK + off16, C::kIdescQK, k > 0);
                }
                mma_commit_elect(&sh.s_full[i]);
                ++s_used;
            };
            for (uint32_t nu = 0; live; ++nu) {
                int32_t idx;
                live = uring_get_warp(sh.ur, nu, idx, abort_flag, err_word, kErrTimeoutBase + 14,
                                      kWaitNs);
                if (!live || idx < 0) break;
                const WlUnit wu = ubase[idx];
                const Unit u = decode_unit(wu, segs);
                const int32_t n = u.ntiles;
                if (n == 0) continue;
                const bool mine = i < u.nsub;
                if (mine) {
                    live = mbar_wait_warp(&sh.q_full[i], q_it & 1, abort_flag, err_word,
                                          kErrTimeoutBase + 3, kWaitNs);
                    if (!live) break;
                }
                {  // stage (K_0)
                    const uint32_t st = kv_it % C::kRingStages;
                    live = mbar_wait_warp(&sh.kv_full[st], (kv_it / C::kRingStages) & 1,
                                          abort_flag, err_word, kErrTimeoutBase + 4, kWaitNs);
                    if (!live) break;
                    if (mine) {
                        issue_qk(st);
                        if (!live) break;
                        if (n == 1) mma_commit_elect(&sh.q_empty[i]);
                    }
                    release(mine, st);
                    ++kv_it;
                }
                for (int32_t j = 0; j < n && live; ++j) {
                    // stage (K_{j+1}, V_j): S_i of tile j+1, then O_i += P_j V_j with P
                    // in two halves of 64 key columns; the stage is released once
                    const uint32_t st = kv_it % C::kRingStages;
                    live = mbar_wait_warp(&sh.kv_full[st], (kv_it / C::kRingStages) & 1,
                                          abort_flag, err_word, kErrTimeoutBase + 5, kWaitNs);
                    if (!live) break;
                    if (mine) {
                        if (j + 1 < n) {
                            issue_qk(st);
                            if (!live) break;
                            if (j + 2 == n) mma_commit_elect(&sh.q_empty[i]);
                        }
                        if (j == 0) {
                            live = mbar_wait_warp(&sh.o_empty[i], (o_cnt & 1) ^ 1, abort_flag,
                                                  err_word, kErrTimeoutBase + 7, kWaitNs);
                            if (!live) break;
                        }
                        const uint64_t dV = dV0 + ((st * C::kStageBytes + C::kTileBytes) >> 4);
                        live = mbar_wait_warp(&sh.p_half[i], p_cnt & 1, abort_flag, err_word,
                                              kErrTimeoutBase + 6, kWaitNs);
                        if (!live) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_elect(tO, tP + k * 8, dV + k * 128, C::kIdescPV,
                                         (j > 0 || k > 0) ? 1u : 0u);
                        live = mbar_wait_warp(&sh.p_full[i], p_cnt & 1, abort_flag, err_word,
                                              kErrTimeoutBase + 12, kWaitNs);
                        if (!live) break;
                        ++p_cnt;
                        tc_fence_after();
#pragma unroll
                        for (int k = 4; k < 8; ++k)
                            mma_ts_elect(tO, tP + k * 8, dV + k * 128, C::kIdescPV, 1u);
                        mma_commit_elect(&sh.pv_done[i]);
                    }
                    release(mine, st);
                    ++kv_it;
                }
                if (!live) break;
                if (mine) {
                    mma_commit_elect(&sh.o_full[i]);
                    ++o_cnt;
                    ++q_it;
                }
            }
            } else {
            for (uint32_t nu = 0; live; ++nu) {
                int32_t idx;
                live = uring_get_warp(sh.ur, nu, idx, abort_flag, err_word, kErrTimeoutBase + 14,
                                      kWaitNs);
                if (!live || idx < 0) break;
                const WlUnit wu = ubase[idx];
                const Unit u = decode_unit(wu, segs);
                const int32_t n = u.ntiles;
                if (n == 0) continue;
                const bool mine = i < u.nsub;
                const bool pair = u.nsub == 2;
                if (mine) {
                    live = mbar_wait_warp(&sh.q_full[i], q_it & 1, abort_flag, err_word,
                                     kErrTimeoutBase + 3, kWaitNs);
                    if (!live) break;
                }
                // prologue: S_i = Q_i K_0^T
                {
                    const uint32_t st = kv_it % C::kStages;
                    live = mbar_wait_warp(&sh.kv_full[st], (kv_it / C::kStages) & 1, abort_flag,
                                     err_word, kErrTimeoutBase + 4, kWaitNs);
                    if (!live) break;
                    live = take_turn(pair);
                    if (!live) break;
                    if (mine) {
                        tc_fence_after();
                        const uint64_t dK = dK0 + ((st * C::kTileBytes) >> 4);
#pragma unroll
                        for (int k = 0; k < D / 16; ++k) {
                            const uint32_t off16 = (k >> 2) * 1024 + (k & 3) * 2;  // bytes >> 4
                            mma_ss_elect(tS, dQ + off16, dK + off16, C::kIdescQK, k > 0);
                        }
                        mma_commit_elect(&sh.s_full[i]);
                        if (n == 1) mma_commit_elect(&sh.q_empty[i]);
                    }
                    pass_turn(pair);
                    release(mine, st);
                    ++kv_it;
                }
                for (int32_t j = 0; j < n && live; ++j) {
                    const bool has_next = j + 1 < n;
                    const uint32_t stv = kv_it % C::kStages;
                    const uint32_t stk = (kv_it + 1) % C::kStages;
                    // Everything that is normally ready early is waited for first,
                    // so that once P_i lands only one wait stands before the MMAs.
                    live = mbar_wait_warp(&sh.kv_full[stv], (kv_it / C::kStages) & 1, abort_flag,
                                          err_word, kErrTimeoutBase + 5, kWaitNs);
                    if (!live) break;
                    if (has_next) {
                        live = mbar_wait_warp(&sh.kv_full[stk], ((kv_it + 1) / C::kStages) & 1,
                                              abort_flag, err_word, kErrTimeoutBase + 8, kWaitNs);
                        if (!live) break;
                    }
                    if (mine && j == 0) {
                        live = mbar_wait_warp(&sh.o_empty[i], (o_cnt & 1) ^ 1, abort_flag,
                                              err_word, kErrTimeoutBase + 7, kWaitNs);
                        if (!live) break;
                    }
                    live = take_turn(pair);
                    if (!live) break;
                    if (mine) {
                        // P_i lands in two halves (key columns [0, 64) and [64, 128));
                        // the first half's MMAs run while the softmax finishes the second
                        const uint64_t dV = dV0 + ((stv * C::kTileBytes) >> 4);
                        live = mbar_wait_warp(&sh.p_half[i], p_cnt & 1, abort_flag, err_word,
                                              kErrTimeoutBase + 6, kWaitNs);
                        if (!live) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_elect(tO, tS + k * 8, dV + k * 128, C::kIdescPV,
                                         (j > 0 || k > 0) ? 1u : 0u);
                        live = mbar_wait_warp(&sh.p_full[i], p_cnt & 1, abort_flag, err_word,
                                              kErrTimeoutBase + 12, kWaitNs);
                        if (!live) break;
                        ++p_cnt;
                        tc_fence_after();
#pragma unroll
                        for (int k = 4; k < 8; ++k)
                            mma_ts_elect(tO, tS + k * 8, dV + k * 128, C::kIdescPV, 1u);
                        if (has_next) {
                            const uint64_t dK = dK0 + ((stk * C::kTileBytes) >> 4);
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint32_t off16 = (k >> 2) * 1024 + (k & 3) * 2;
                                mma_ss_elect(tS, dQ + off16, dK + off16, C::kIdescQK, k > 0);
                            }
                            mma_commit_elect(&sh.s_full[i]);
                            if (j + 2 == n) mma_commit_elect(&sh.q_empty[i]);
                        }
                    }
                    pass_turn(pair);
                    release(mine, stv);
                    if (has_next) release(mine, stk);
                    kv_it += has_next ? 2 : 1;
                }
                if (!live) break;
                if (mine) {
                    mma_commit_elect(&sh.o_full[i]);
                    ++o_cnt;
                    ++q_it;
                }
            }
            }
            // drain every MMA this thread issued before tensor memory is freed
            mma_commit_elect(&sh.done[i]);
            mbar_wait_drain(&sh.done[i], 0, kDrainNs);
        }
        __syncwarp();
      }
      finish();
      return;
    } else {
        regs_alloc<Regs<D>::kSoftmax>();
        // ------------------------------------------------------- softmax / epilogue
        const int i = (warp - 4) >> 2;           // sub-tile of this warpgroup
        const int r = (warp & 3) * 32 + lane;    // query row = tensor-memory lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + i * 128;
        const uint32_t tO = tmem + lane_base + 256 + i * 128;
        uint32_t s_cnt = 0, o_cnt = 0;
        bool live = true;
        // The roles take unit n from the producer's ring; the softmax takes the
        // next one before its epilogue (the producer published it once it had
        // issued this unit's loads), so that the unit's description is read from
        // global memory while the epilogue runs.
        int32_t idx = -1;
        WlUnit wu;
        auto take_unit = [&](uint32_t n) {
            live = uring_get(sh.ur, n, idx, abort_flag, err_word, kErrTimeoutBase + 14, kWaitNs);
            if (live && idx >= 0) wu = ubase[idx];
        };
        // The epilogue of a unit (O / l and the LSE out) runs after the softmax of
        // the next unit's first kv tile has handed its P over, so that the tensor
        // pipe computes that tile's PV and the next QK meanwhile instead of
        // waiting for the stores (or during a unit without tiles for this
        // sub-tile, which would leave its warps idle).  pst, pm,
        // pl: the pending unit's sub-tile and its running max and sum.  The fused
        // ring step (ACC: read-modify-write of the running fp32 O and LSE) runs its
        // epilogue at once: deferred, it measured slower.
        bool pend = false;
        SubTile pst{0, 0, 0, 0};
        float pm = 0.f, pl = 0.f;
        auto epilogue = [&]() {
            pend = false;
            live = mbar_wait(&sh.o_full[i], o_cnt & 1, abort_flag, err_word, kErrTimeoutBase + 10,
                             kWaitNs);
            if (!live) return;
            ++o_cnt;
            const SubTile& st = pst;
            const bool valid = r < st.nrows;
            const float m_used = pm, l_sum = pl;
            tc_fence_after();
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            const int64_t row = (int64_t)(st.q_row + r) * p.hq + st.head;
            // read the whole row of O, hand the tensor memory back to the MMA
            // warp, then normalise and store
            uint32_t o[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + c * 32, o[c]);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
            tc_fence_before();
            mbar_arrive(&sh.o_empty[i]);
            const float lse_new =
                l_sum > 0.f ? (m_used + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
            float* lrow = p.lse + (int64_t)st.head * p.q_tokens + st.q_row + r;
            // every row of this warp belongs to the sub-tile (warp-uniform)
            const bool warp_full = __all_sync(0xffffffffu, valid);
            if constexpr (ACC) {
              if (valid) {
                // fused ring step: merge this partial into the running fp32 (O, LSE)
                //   lse = ln(e^lse_run + e^lse_new),
                //   O = e^(lse_run - lse) O_run + e^(lse_new - lse) O_new
                // a row without keys here (lse_new = -inf) keeps its running values
                if (lse_new != -INFINITY) {
                    const float lse_old = *lrow;
                    const float mx = fmaxf(lse_old, lse_new);
                    const float ea = lse_old == -INFINITY ? 0.f : expf(lse_old - mx);
                    const float eb = expf(lse_new - mx);
                    const float wa = ea / (ea + eb), wb = eb / (ea + eb) * inv;
                    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * D);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            // a running value never merged before may be anything
                            const float4 x = ea == 0.f ? make_float4(0.f, 0.f, 0.f, 0.f)
                                                       : dst[c * 8 + e];
                            dst[c * 8 + e] =
                                make_float4(wa * x.x + wb * __uint_as_float(o[c][4 * e]),
                                            wa * x.y + wb * __uint_as_float(o[c][4 * e + 1]),
                                            wa * x.z + wb * __uint_as_float(o[c][4 * e + 2]),
                                            wa * x.w + wb * __uint_as_float(o[c][4 * e + 3]));
                        }
                    }
                    *lrow = mx + logf(ea + eb);
                }
              }
            } else if (warp_full) {
                // all 32 rows of this warp belong to the sub-tile: stage them in shared
                // memory, 128 bytes of every row at a time (128-byte swizzle: 16-byte
                // chunk k of row `lane` at (k ^ (lane % 8)) * 16), and write each 32-row
                // block with one TMA store, so that the stores leave the warp as whole
                // rows instead of one 16-byte piece of 32 different rows per instruction
                uint8_t* stg = sStage + (warp - 4) * 4096;
                const uint32_t row_addr = smem_u32(stg) + lane * 128;
                const int32_t row0 = st.q_row + (warp & 3) * 32;
                if (p.out_fp32) {
#pragma unroll
                    for (int cb = 0; cb < D / 32; ++cb) {
                        if (lane == 0) bulk_wait_read_all();  // the buffer's last store has read it
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            st_shared_v4(row_addr + ((k ^ (lane & 7)) << 4),
                                         __float_as_uint(__uint_as_float(o[cb][4 * k]) * inv),
                                         __float_as_uint(__uint_as_float(o[cb][4 * k + 1]) * inv),
                                         __float_as_uint(__uint_as_float(o[cb][4 * k + 2]) * inv),
                                         __float_as_uint(__uint_as_float(o[cb][4 * k + 3]) * inv));
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tmo, stg, cb * 32, st.head, row0);
                            bulk_commit_group();
                        }
                    }
                } else {
#pragma unroll
                    for (int cb = 0; cb < D / 64; ++cb) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t* v = &o[2 * cb + (k >> 2)][(k & 3) * 8];
                            st_shared_v4(row_addr + ((k ^ (lane & 7)) << 4),
                                         pack_bf16x2(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                                         pack_bf16x2(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                                         pack_bf16x2(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                                         pack_bf16x2(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tmo, stg, cb * 64, st.head, row0);
                            bulk_commit_group();
                        }
                    }
                }
                *lrow = lse_new;
            } else if (valid) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    if (p.out_fp32) {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) +
                                                                row * D + c * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(o[c][4 * e]) * inv,
                                                 __uint_as_float(o[c][4 * e + 1]) * inv,
                                                 __uint_as_float(o[c][4 * e + 2]) * inv,
                                                 __uint_as_float(o[c][4 * e + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(
                            reinterpret_cast<__nv_bfloat16*>(p.out) + row * D + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(
                                pack_bf16x2(__uint_as_float(o[c][8 * e]) * inv, __uint_as_float(o[c][8 * e + 1]) * inv),
                                pack_bf16x2(__uint_as_float(o[c][8 * e + 2]) * inv, __uint_as_float(o[c][8 * e + 3]) * inv),
                                pack_bf16x2(__uint_as_float(o[c][8 * e + 4]) * inv, __uint_as_float(o[c][8 * e + 5]) * inv),
                                pack_bf16x2(__uint_as_float(o[c][8 * e + 6]) * inv, __uint_as_float(o[c][8 * e + 7]) * inv));
                    }
                }
                *lrow = lse_new;
            }
        };
        take_unit(0);
        for (uint32_t nu = 0; live && idx >= 0; ++nu) {
            const Unit u = decode_unit(wu, segs);
            if (i >= u.nsub || u.ntiles == 0) {
                // this sub-tile has no tiles here: the pending epilogue runs now
                if (!ACC && pend) epilogue();
                if (!live) break;
                // no key for these rows: O = 0, LSE = -inf, which a running
                // (O, LSE) absorbs unchanged
                if (i < u.nsub && !ACC) write_empty_rows(p, u.st[i], r, D);
                take_unit(nu + 1);
                continue;
            }
            const SubTile st = i == 0 ? u.st[0] : u.st[1];
            const bool valid = r < st.nrows;
            const int32_t q_pos = st.q_pos + r;
            if (ACC && valid) {
                // the epilogue reads this row's running O and LSE back: start moving
                // them from DRAM to L2 now, so that the read does not wait on DRAM
                const float* orow =
                    reinterpret_cast<const float*>(p.out) + ((int64_t)(st.q_row + r) * p.hq + st.head) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) prefetch_l2(orow + c * 32);
                prefetch_l2(p.lse + (int64_t)st.head * p.q_tokens + st.q_row + r);
            }
            float m_used = -INFINITY, l_sum = 0.f;
            for (int32_t rr = 0; rr < u.run_count && live; ++rr) {
                const WlRun run = runs[u.run_begin + rr];
                const WlSlice s = slices[run.slice];
                // allowed keys of this row, relative to the slice's first key:
                // [lim_lo, lim_hi) (by the slice's MaskType; nothing for padding rows)
                int64_t klo, khi;
                slice_keys_of_query(s, q_pos, klo, khi, slice_mask(p.wl, h, s, run.slice));
                const int32_t lim_hi = valid ? (int32_t)khi : 0;
                const int32_t lim_lo = (int32_t)klo;
                for (int32_t jt = run.lo; jt < run.hi && live; ++jt) {
                    // allowed columns [c_lo, c_hi) in this kv tile, settled while S
                    // is still being computed
                    const int32_t kt0 = jt * 128;
                    const int32_t c_hi = min(128, lim_hi - kt0), c_lo = max(0, lim_lo - kt0);
                    const bool need_mask = __any_sync(0xffffffffu, c_lo > 0 || c_hi < 128);
                    live = mbar_wait(&sh.s_full[i], s_cnt & 1, abort_flag, err_word,
                                     kErrTimeoutBase + 9, kWaitNs);
                    if (!live) break;
                    ++s_cnt;
                    tc_fence_after();
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
                    if (C::kSplitP) {
                        // S_i has been read: QK of the next kv tile may overwrite it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh.s_free[i]);
                    }
                    if (need_mask) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int col = c * 32 + e;
                                if (col < c_lo || col >= c_hi) sr[c][e] = __float_as_uint(-INFINITY);
                            }
                    }
                    // row max: 16 partial maxima over 8 columns each (3-input max), then
                    // a 3-input tree; 7 dependent steps instead of one long chain
                    float pm[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const uint32_t* v = &sr[q >> 2][(q & 3) * 8];
                        float m3 = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]),
                                         __uint_as_float(v[2]));
                        m3 = fmax3(m3, __uint_as_float(v[3]), __uint_as_float(v[4]));
                        m3 = fmax3(m3, __uint_as_float(v[5]), __uint_as_float(v[6]));
                        pm[q] = fmaxf(m3, __uint_as_float(v[7]));
                    }
                    const float t0 = fmax3(pm[0], pm[1], pm[2]), t1 = fmax3(pm[3], pm[4], pm[5]);
                    const float t2 = fmax3(pm[6], pm[7], pm[8]), t3 = fmax3(pm[9], pm[10], pm[11]);
                    const float t4 = fmax3(pm[12], pm[13], pm[14]);
                    const float mx = fmaxf(fmax3(t0, t1, t2), fmax3(t3, t4, pm[15]));
                    const float m_tile = mx * p.scale_log2;  // -inf stays -inf
                    // Lazy rescaling: the reference maximum moves only when this tile's
                    // maximum exceeds it by more than the threshold (or it is still -inf,
                    // when O and l are zero and need no rescale).
                    if (C::kSplitP && s_cnt >= 2) {
                        // O and the P columns: PV of the previous tile must be complete
                        live = mbar_wait(&sh.pv_done[i], (s_cnt - 2) & 1, abort_flag, err_word,
                                         kErrTimeoutBase + 16, kWaitNs);
                        if (!live) break;
                        tc_fence_after();
                    }
                    float alpha = 1.f;
                    bool rescale = false;
                    if (m_tile > m_used + kRescaleThreshold) {
                        rescale = m_used != -INFINITY;
                        if (rescale) alpha = ex2_approx(m_used - m_tile);
                        m_used = m_tile;
                    }
                    l_sum *= alpha;
                    // rare: the running max moved, rescale this row of O first (PV of
                    // the previous tile has completed: it ran before QK of this one, or
                    // with P apart from S, pv_done said so)
                    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + c * 32, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tO + c * 32, o);
                        }
                    }
                    // P = 2^(s*scale*log2e - m), packed to bf16 pairs in place
                    // (pair e/2 lands in a register already consumed), handed to
                    // the MMA warp in two halves of 64 key columns
                    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
                    // packed fp32x2 FMA / add: two elements per instruction
                    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nm2 = make_float2(neg_m, neg_m);
                    float2 part[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        part[c] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])),
                                sl2, nm2);
                            const float p0 = ex2_approx(x.x);
                            const float p1 = ex2_approx(x.y);
                            part[c] = __fadd2_rn(part[c], make_float2(p0, p1));
                            sr[c][e >> 1] = pack_bf16x2(p0, p1);
                        }
                        // the first half is announced after chunk 2's exponentials, so
                        // that the wait for its stores overlaps them
                        if (c == 2) {
                            tmem_st_wait();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.p_half[i]);
                        }
                        tmem_st16((C::kSplitP ? tO + 64 : tS) + c * 16, sr[c]);
                        if (c == 3) {
                            tmem_st_wait();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.p_full[i]);
                        }
                    }
                    const float2 ps = __fadd2_rn(__fadd2_rn(part[0], part[1]), __fadd2_rn(part[2], part[3]));
                    l_sum += ps.x + ps.y;
                    if (!ACC && pend) {
                        epilogue();
                        if (!live) break;
                    }
                }
            }
            if (!live) break;
            take_unit(nu + 1);
            if (!live) break;
            pend = true;
            pst = st;
            pm = m_used;
            pl = l_sum;
            if constexpr (ACC) {
                epilogue();
                if (!live) break;
            }
        }
        if (!ACC && live && pend) epilogue();
        finish();
    }

}

}  // namespace
}  // namespace pva

// ------------------------------------------------------------------ host side
namespace pva {
namespace {

std::atomic<int32_t> g_withhold_kv{0};  // pva_debug_withhold_kv_load

template <int D>
pva_status launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                  const CUtensorMap& mo, const AttnParams& ap, cudaStream_t st) {
    auto kern = ap.accumulate ? attn_fwd_kernel<D, true> : attn_fwd_kernel<D, false>;
    // setmaxnreg.inc draws from the registers the block was launched with: the
    // split must fit in (threads x registers per thread) or the increase would
    // never be granted.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PVA_ERR_CUDA;
    if ((int64_t)fa.numRegs * kThreads <
        128 * (int64_t)Regs<D>::kCtrl + 256 * (int64_t)Regs<D>::kSoftmax)
        return PVA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem) !=
        cudaSuccess)
        return PVA_ERR_CUDA;
    kern<<<ap.num_ctas, kThreads, Cfg<D>::kSmem, st>>>(mq, mk, mv, mo, ap);
    return cudaGetLastError() == cudaSuccess ? PVA_OK : PVA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pva

using namespace pva;

namespace {

pva_status attn_fwd_impl(const void* q, const void* k, const void* v,
                         const int32_t* cu_seqlens_dev, const pva_mask_desc* mask,
                         const pva_worklist_params* params, int32_t head_dim,
                         const void* worklist_dev, void* out, int32_t out_is_fp32, float* lse,
                         float softmax_scale, uint64_t* cta_busy_ns, int32_t accumulate,
                         void* stream) {
    if (!mask || !params || !worklist_dev) return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens == 0 && mask->k_tokens >= 0) return PVA_OK;  // no query row: nothing to do
    if (!out || !lse || !q) return PVA_ERR_INVALID_ARG;
    if (mask->kind != PVA_MASK_SLICES && !cu_seqlens_dev) return PVA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PVA_ERR_UNSUPPORTED;
    if (params->tile_m != 128 || params->tile_n != 128) return PVA_ERR_UNSUPPORTED;
    if (params->num_q_heads <= 0 || params->num_kv_heads <= 0 ||
        params->num_q_heads % params->num_kv_heads != 0)
        return PVA_ERR_INVALID_ARG;
    if (out_is_fp32 != 0 && out_is_fp32 != 1) return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens < 0 || mask->k_tokens < 0) return PVA_ERR_INVALID_ARG;
    if (mask->k_tokens > 0 && (!k || !v)) return PVA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(lse) ||
        (mask->k_tokens > 0 && (!aligned16(k) || !aligned16(v))) ||
        (reinterpret_cast<uintptr_t>(worklist_dev) & 255u))
        return PVA_ERR_INVALID_ARG;
    const int32_t nc = resolve_num_ctas(params->num_ctas);
    if (nc <= 0) return PVA_ERR_CUDA;
    if (nc > kMaxBins) return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens == 0) return PVA_OK;
    CUtensorMap mq, mk, mv, mo;
    const void* kp = mask->k_tokens > 0 ? k : q;  // no key rows: maps are never read
    const void* vp = mask->k_tokens > 0 ? v : q;
    const int32_t kh = mask->k_tokens > 0 ? params->num_kv_heads : params->num_q_heads;
    if (!make_map(&mq, q, mask->q_tokens, params->num_q_heads, head_dim) ||
        !make_map(&mk, kp, mask->k_tokens, kh, head_dim) ||
        !make_map(&mv, vp, mask->k_tokens, kh, head_dim) ||
        !make_map(&mo, out, mask->q_tokens, params->num_q_heads, head_dim, 32,
                  out_is_fp32 ? 4 : 2))
        return PVA_ERR_CUDA;
    AttnParams ap;
    ap.wl = reinterpret_cast<const uint8_t*>(worklist_dev);
    ap.out = out;
    ap.lse = lse;
    ap.busy = cta_busy_ns;
    ap.q_tokens = mask->q_tokens;
    ap.k_tokens = mask->k_tokens;
    ap.hq = params->num_q_heads;
    ap.hkv = params->num_kv_heads;
    ap.out_fp32 = out_is_fp32;
    ap.accumulate = accumulate;
    ap.num_ctas = nc;
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.withhold_kv = g_withhold_kv.load(std::memory_order_relaxed);
    ap.dynamic = params->dispatch == PVA_DISPATCH_STATIC ? 0 : 1;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return head_dim == 128 ? launch<128>(mq, mk, mv, mo, ap, st)
                           : launch<64>(mq, mk, mv, mo, ap, st);
}

}  // namespace

extern "C" pva_status pva_attn_fwd(const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens_dev, const pva_mask_desc* mask,
                                   const pva_worklist_params* params, int32_t head_dim,
                                   const void* worklist_dev, void* out, int32_t out_is_fp32,
                                   float* lse, float softmax_scale, uint64_t* cta_busy_ns,
                                   void* stream) {
    return attn_fwd_impl(q, k, v, cu_seqlens_dev, mask, params, head_dim, worklist_dev, out,
                         out_is_fp32, lse, softmax_scale, cta_busy_ns, 0, stream);
}

extern "C" pva_status pva_attn_fwd_accumulate(const void* q, const void* k, const void* v,
                                              const int32_t* cu_seqlens_dev,
                                              const pva_mask_desc* mask,
                                              const pva_worklist_params* params,
                                              int32_t head_dim, const void* worklist_dev,
                                              float* o_run, float* lse_run, float softmax_scale,
                                              uint64_t* cta_busy_ns, void* stream) {
    return attn_fwd_impl(q, k, v, cu_seqlens_dev, mask, params, head_dim, worklist_dev, o_run, 1,
                         lse_run, softmax_scale, cta_busy_ns, 1, stream);
}

extern "C" void pva_debug_withhold_kv_load(int32_t enable) {
    g_withhold_kv.store(enable != 0 ? 1 : 0, std::memory_order_relaxed);
}
