// noalloc.cu -- attention forward for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: a plugin inside a runtime that owns a fixed device
// memory pool, a serving process whose memory budget is fixed up front, or a
// plain C host that links only this library and has no device allocator of
// its own.  pva_attn_fwd_noalloc needs from them only the inputs
// and outputs: the worklist it builds lives in a file-scope device array of
// fixed size (kNoAllocScratchBytes) that every GPU loading the library holds
// until the process exits.
//
// When the array's memory is committed depends on how CUDA loads modules:
// with lazy loading (the default) the driver loads this module, and commits
// the 16 MiB, at the first cudaGetSymbolAddress, i.e. inside the first call
// on a device.  A caller with a fixed memory budget makes one warm-up call
// at start-up, before it fixes the budget and before any stream capture.
//
// The host side cannot use the array's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and caches it together with the CUDA context it
// belongs to; a new context on that device (after cudaDeviceReset, say) is
// looked up again.  All calls on a device share the array and it keeps the
// previous call's contents; the worklist build rewrites its header (error
// word, counts, sums) before anything reads it, so nothing has to be cleared.
// Two calls that overlap on the GPU (different streams, or host threads
// without ordering) race on the array.  Device-side failures of the last call
// (bad cu_seqlens, a capacity overflow, a wait that timed out) are read with
// pva_noalloc_error.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pva.h"

namespace pva {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Driver entry points, looked up once (the runtime is linked statically; the
// driver library is resolved at run time).
template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(f);
    return nullptr;
}

// Unique id of the current CUDA context (0: none is current).
bool current_ctx_id(unsigned long long* id) {
    static CtxGetCurrentFn get = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device: looked up on
// the first call per device, and again if the device's context changed.
pva_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PVA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PVA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long ctx = 0;
    if (!current_ctx_id(&ctx)) return PVA_ERR_CUDA;
    if (ctx != 0 && g_scratch_ptr[dev] && g_scratch_ctx[dev] == ctx) {
        *out = g_scratch_ptr[dev];
        return PVA_OK;
    }
    // (the runtime makes the device's primary context current here if no
    // context was current yet)
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PVA_ERR_CUDA;
    if (!current_ctx_id(&ctx) || ctx == 0) return PVA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
    *out = ptr;
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

extern "C" pva_status pva_noalloc_error(int32_t* code_out, void* stream) {
    if (!code_out) return PVA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const pva_status st = pva::scratch_for_current_device(&scratch);
    if (st != PVA_OK) return st;
    return pva_worklist_error(scratch, code_out, stream);
}
