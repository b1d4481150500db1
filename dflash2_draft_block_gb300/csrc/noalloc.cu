// dflash2_unary_topk_noalloc: unary_topk for callers that cannot allocate device
// memory.
//
// Some callers run inside a host framework that owns every device allocation
// and forbids new ones while it executes a step (an engine plugin, an embedded
// runtime with a fixed memory budget), or sit on a latency-critical path where a
// cudaMalloc, which may synchronise the device, is not acceptable.  They cannot
// size and allocate the workspace dflash2_unary_topk asks for.  This entry point
// takes the same inputs and outputs but uses a scratch array that lives in the
// library itself: a file-scope __device__ array of DF2_NOALLOC_SCRATCH_BYTES,
// which every GPU that loads the library holds until the process exits.
//
// The scratch holds the per-CTA candidate lists the top-K merge reads; every slot
// the merge reads is written earlier in the same call, so nothing has to start
// at zero and the contents left by the previous call do no harm.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DF2_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the array.  In host code the array's
// name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DF2_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DF2_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return DF2_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DF2_OK;
}

}  // namespace

DF2_API int dflash2_unary_topk_noalloc(const uint16_t* h, int64_t P, int64_t D,
                                       const uint16_t* W_lm, int64_t V, int K, float output_multiplier,
                                       float final_logit_softcapping, const uint16_t* W_H, int r,
                                       float* G, int32_t* topk_ids,
                                       float* topk_vals, int32_t* dev_status, void* stream) {
    const size_t need = dflash2_unary_topk_workspace_size(P, D, V, K, r);
    if (need > DF2_NOALLOC_SCRATCH_BYTES) return DF2_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        // the scratch address is per device: a stream of another device would
        // have its kernels read this device's address
        if (stream != nullptr) {
            int dev = 0, sdev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
                return DF2_ERR_CUDA;
            if (sdev != dev) return DF2_ERR_INVALID_ARGUMENT;
        }
        const int rc = scratch_for_current_device(&scratch);
        if (rc != DF2_OK) return rc;
    }
    return dflash2_unary_topk(h, P, D, W_lm, V, K, output_multiplier, final_logit_softcapping, W_H, r, G,
                              topk_ids, topk_vals, scratch,
                              scratch ? DF2_NOALLOC_SCRATCH_BYTES : 0, dev_status, stream);
}
