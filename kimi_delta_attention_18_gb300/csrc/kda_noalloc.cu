// Prefill for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// prefill: plugins of inference engines that hand out all device memory up
// front and forbid allocation while work is enqueued, or hosts whose memory is
// owned entirely by another framework's pool.  kda_prefill_chunked needs a
// workspace when it splits sequences into segments; this entry point supplies
// that workspace from a fixed array compiled into the library instead, so the
// caller passes only its inputs and outputs.
//
// The array lives in device memory on every GPU that loads the library and is
// held until the process exits.  It is shared by every call on a device and
// keeps whatever the last call left in it; nothing in it has to start at zero
// (every slot the prefill reads is written earlier in the same call), but two
// calls that overlap on the GPU (different streams, no ordering between them)
// race on it and corrupt each other's results.
#include <mutex>

#include "kda_internal.cuh"

namespace {

// The scratch itself.  In host code `g_noalloc_scratch` is only a stand-in
// symbol, not a device address: its device address comes from
// cudaGetSymbolAddress, once per device, below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up on the first
// call made with that device current.
kda_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_prefill_chunked_noalloc(const kda_prefill_desc_t *desc,
                                                    const void *q, const void *k, const void *v,
                                                    const float *g, const float *beta,
                                                    const float *S0, const int32_t *cu_seqlens,
                                                    void *out, float *S_final,
                                                    int32_t *dev_status, void *stream) {
    if (!desc) return KDA_ERR_INVALID_ARG;
    const size_t need = kda_prefill_workspace_size(desc);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const kda_status_t rc = scratch_on_current_device(&scratch);
        if (rc != KDA_OK) return rc;
    }
    return kda_prefill_chunked(desc, q, k, v, g, beta, S0, cu_seqlens, out, S_final, scratch,
                               need > 0 ? (size_t)KDA_NOALLOC_SCRATCH_BYTES : 0, dev_status,
                               stream);
}
