// host_io.cu -- the forward pass for callers whose inputs and results live in
// host memory: the copies in, the worklist build, the attention and the
// copies out, enqueued in that order on one stream.
//
// Callers that stream many packs alternate two streams, each with its own
// device buffers, so that one pack's copies in overlap the previous pack's
// attention and copies out (host-to-device and device-to-host copies use
// separate copy engines).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pva.h"

extern "C" pva_status pva_attn_fwd_host(const void* q_host, const void* k_host,
                                        const void* v_host, const int32_t* cu_seqlens_host,
                                        int32_t num_docs, const pva_mask_desc* mask,
                                        const pva_worklist_params* params, int32_t head_dim,
                                        void* out_host, float* lse_host, float softmax_scale,
                                        void* q_dev, void* k_dev, void* v_dev,
                                        int32_t* cu_seqlens_dev, void* worklist_dev,
                                        size_t worklist_bytes, void* out_dev, float* lse_dev,
                                        void* stream) {
    if (!mask || !params || !q_host || !q_dev || !out_host || !out_dev || !lse_host || !lse_dev)
        return PVA_ERR_INVALID_ARG;
    if (mask->q_tokens < 0 || mask->k_tokens < 0 || num_docs < 0 || params->num_q_heads <= 0 ||
        params->num_kv_heads <= 0 || (head_dim != 64 && head_dim != 128))
        return PVA_ERR_INVALID_ARG;
    const bool need_cu = mask->kind != PVA_MASK_SLICES;
    if (need_cu && (!cu_seqlens_host || !cu_seqlens_dev)) return PVA_ERR_INVALID_ARG;
    if (mask->k_tokens > 0 && (!k_host || !v_host || !k_dev || !v_dev)) return PVA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t qb = (size_t)mask->q_tokens * params->num_q_heads * head_dim * 2;
    const size_t kb = (size_t)mask->k_tokens * params->num_kv_heads * head_dim * 2;
    const size_t lb = (size_t)mask->q_tokens * params->num_q_heads * 4;
    // one cudaMemcpyAsync per buffer
    if (cudaMemcpyAsync(q_dev, q_host, qb, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return PVA_ERR_CUDA;
    if (kb > 0 && (cudaMemcpyAsync(k_dev, k_host, kb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
                   cudaMemcpyAsync(v_dev, v_host, kb, cudaMemcpyHostToDevice, st) != cudaSuccess))
        return PVA_ERR_CUDA;
    if (need_cu && cudaMemcpyAsync(cu_seqlens_dev, cu_seqlens_host, ((size_t)num_docs + 1) * 4,
                                   cudaMemcpyHostToDevice, st) != cudaSuccess)
        return PVA_ERR_CUDA;
    pva_status s = pva_build_worklist(need_cu ? cu_seqlens_dev : nullptr, num_docs, mask, params,
                                      worklist_dev, worklist_bytes, stream);
    if (s != PVA_OK) return s;
    s = pva_attn_fwd(q_dev, k_dev, v_dev, need_cu ? cu_seqlens_dev : nullptr, mask, params,
                     head_dim, worklist_dev, out_dev, 0, lse_dev, softmax_scale, nullptr, stream);
    if (s != PVA_OK) return s;
    if (cudaMemcpyAsync(out_host, out_dev, qb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(lse_host, lse_dev, lb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PVA_ERR_CUDA;
    return PVA_OK;
}
