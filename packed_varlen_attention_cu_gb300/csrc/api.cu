// api.cu -- host-only entry points of the C ABI: status strings, version,
// zigzag shard sizes.
#include <stdint.h>

#include "../../include/pva.h"

extern "C" const char* pva_status_string(pva_status status) {
    switch (status) {
    case PVA_OK: return "ok";
    case PVA_ERR_INVALID_ARG: return "invalid argument";
    case PVA_ERR_BUFFER_TOO_SMALL: return "worklist buffer too small";
    case PVA_ERR_CUDA: return "CUDA call failed";
    case PVA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PVA_ERR_TIMEOUT: return "device-side wait timed out";
    case PVA_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

extern "C" int32_t pva_version(void) { return 10000; }  // 1.0.0

// Rows of zigzag shard `rank`: per document, chunk c holds floor(l/2cp)
// tokens plus one if c < l mod 2cp; the rank owns chunks rank and 2cp-1-rank.
extern "C" int32_t pva_zigzag_shard_len(const int32_t* cu_seqlens_host, int32_t num_docs,
                                        int32_t cp, int32_t rank) {
    if (!cu_seqlens_host || num_docs < 0 || cp < 1 || rank < 0 || rank >= cp) return -1;
    if (cu_seqlens_host[0] != 0) return -1;
    int64_t total = 0;
    const int32_t n = 2 * cp;
    for (int32_t d = 0; d < num_docs; ++d) {
        const int32_t len = cu_seqlens_host[d + 1] - cu_seqlens_host[d];
        if (len < 0) return -1;
        const int32_t base = len / n, rem = len % n;
        total += base + (rank < rem ? 1 : 0);
        total += base + ((n - 1 - rank) < rem ? 1 : 0);
    }
    return total > INT32_MAX ? -1 : (int32_t)total;
}
