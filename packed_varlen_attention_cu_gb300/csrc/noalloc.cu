// noalloc.cu -- attention forward for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: a plugin inside a runtime that owns a fixed device
// memory pool, a serving process whose memory budget is fixed up front, or a
// plain C host that links only this library and has no device allocator of
// its own.  pva_attn_fwd_noalloc needs from them only the inputs
// and outputs: the worklist it builds lives in a file-scope device array of
// fixed size (kNoAllocScratchBytes), allocated once when the library's module
// is loaded on a device and kept until the process exits.
//
// The host side cannot use the array's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and caches it; that first call should therefore
// come before any stream capture.  All calls on a device share the array and
// it keeps the previous call's contents; the worklist build rewrites its
// header (error word, counts, sums) before anything reads it, so nothing has
// to be cleared.  Two calls that overlap on the GPU (different streams, or
// host threads without ordering) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pva.h"

namespace pva {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
pva_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PVA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PVA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return PVA_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PVA_OK;
}

}  // namespace
}  // namespace pva

extern "C" size_t pva_noalloc_scratch_bytes(void) { return pva::kNoAllocScratchBytes; }

extern "C" pva_status pva_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                           const int32_t* cu_seqlens_dev, int32_t num_docs,
                                           const pva_mask_desc* mask,
                                           const pva_worklist_params* params, int32_t head_dim,
                                           void* out, int32_t out_is_fp32, float* lse,
                                           float softmax_scale, void* stream) {
    if (!mask || !params) return PVA_ERR_INVALID_ARG;
    const size_t need = pva_worklist_bytes(num_docs, mask, params);
    if (need == 0) return PVA_ERR_INVALID_ARG;
    if (need > pva::kNoAllocScratchBytes) return PVA_ERR_BUFFER_TOO_SMALL;
    void* scratch = nullptr;
    const pva_status st = pva::scratch_for_current_device(&scratch);
    if (st != PVA_OK) return st;
    const pva_status b = pva_build_worklist(cu_seqlens_dev, num_docs, mask, params, scratch,
                                            pva::kNoAllocScratchBytes, stream);
    if (b != PVA_OK) return b;
    return pva_attn_fwd(q, k, v, cu_seqlens_dev, mask, params, head_dim, scratch, out,
                        out_is_fp32, lse, softmax_scale, nullptr, stream);
}
