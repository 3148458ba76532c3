// unit_feed.cuh -- how a persistent CTA's roles learn which work unit comes next.
//
// One producer thread decides the CTA's next unit and publishes its index in
// a small shared-memory ring (UnitRing); every other role reads the slots in
// the same order and releases each after reading it.  The index is -1 once
// the CTA has no more work.  The producer decides either from a fixed list
// (static dispatch) or by claiming the next rank of a dispatch order from a
// global counter (dynamic dispatch: "数据并行负载均衡" §4.4's LPT rule with the
// least loaded worker being whichever CTA frees up first).
//
// A dispatch counter is a pair (next, done) in device memory that starts at
// (0, 0): CTAs claim ranks with atomicAdd on `next`, and at exit each CTA adds
// one to `done`; the last one puts both back to 0, so the next launch that
// uses the same counter starts from rank 0.  One launch at a time may use a
// counter (launches ordered on a stream are fine).
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace pva {

template <int R>
struct UnitRing {
    uint64_t full[R], empty[R];
    int32_t slot[R];
};

// `readers` arrivals free a slot.
template <int R>
__device__ __forceinline__ void uring_init(UnitRing<R>& r, uint32_t readers) {
    for (int s = 0; s < R; ++s) {
        mbar_init(&r.full[s], 1);
        mbar_init(&r.empty[s], readers);
    }
}

// Producer: slot n (the n-th unit of this CTA) is free once every reader has
// taken unit n - R.
template <int R>
__device__ __forceinline__ bool uring_wait_free(UnitRing<R>& r, uint32_t n,
                                                volatile int* abort_flag, int* err_word, int site,
                                                uint64_t timeout_ns) {
    return mbar_wait(&r.empty[n % R], ((n / R) & 1) ^ 1, abort_flag, err_word, site, timeout_ns);
}

// Producer: publish unit index `idx` (-1: no more work) as the n-th unit.
template <int R>
__device__ __forceinline__ void uring_put(UnitRing<R>& r, uint32_t n, int32_t idx) {
    r.slot[n % R] = idx;
    mbar_arrive(&r.full[n % R]);  // release: the slot write is seen by the readers
}

// A whole converged warp takes the n-th unit (one arrival for the warp).
template <int R>
__device__ __forceinline__ bool uring_get_warp(UnitRing<R>& r, uint32_t n, int32_t& idx,
                                               volatile int* abort_flag, int* err_word, int site,
                                               uint64_t timeout_ns) {
    if (!mbar_wait_warp(&r.full[n % R], (n / R) & 1, abort_flag, err_word, site, timeout_ns))
        return false;
    idx = *reinterpret_cast<volatile int32_t*>(&r.slot[n % R]);
    __syncwarp();
    mbar_arrive_elect(&r.empty[n % R]);
    return true;
}

// One thread takes the n-th unit (one arrival per thread).
template <int R>
__device__ __forceinline__ bool uring_get(UnitRing<R>& r, uint32_t n, int32_t& idx,
                                          volatile int* abort_flag, int* err_word, int site,
                                          uint64_t timeout_ns) {
    if (!mbar_wait(&r.full[n % R], (n / R) & 1, abort_flag, err_word, site, timeout_ns))
        return false;
    idx = *reinterpret_cast<volatile int32_t*>(&r.slot[n % R]);
    mbar_arrive(&r.empty[n % R]);
    return true;
}

// Dynamic dispatch: the next rank for this CTA.
__device__ __forceinline__ int32_t dispatch_claim(int32_t* next) { return atomicAdd(next, 1); }

// Called by one thread of every CTA after its last claim (all of its roles
// are done): the last CTA of the launch resets the counter.
__device__ __forceinline__ void dispatch_exit(int32_t* next, int32_t* done) {
    __threadfence();
    if (atomicAdd(done, 1) == (int)gridDim.x - 1) {
        atomicExch(next, 0);
        atomicExch(done, 0);
    }
}

}  // namespace pva
