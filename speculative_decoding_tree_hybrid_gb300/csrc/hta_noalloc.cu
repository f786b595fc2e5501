// hta_verify_noalloc: hta_verify for callers that cannot allocate device
// memory, such as code running while a CUDA graph is being captured with an
// allocator that forbids new allocations, inference servers whose memory pool
// is fixed up front, or plug-ins that only receive tensors from a host
// framework. Instead of a caller-provided workspace, the split-KV partials and
// the grid-barrier counters live in the fixed array below, which every GPU
// that loads this library keeps until the process exits.
#include <mutex>

#include "../../include/hta.h"

namespace {

// file-scope scratch; its device address is fetched once per device
static __device__ __align__(256) unsigned char g_scratch[HTA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up on the first
// call for that device, with that device current). nullptr on failure.
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" hta_status hta_verify_noalloc(const hta_dims *dims, const hta_bf16 *q, const hta_bf16 *k_cache,
                                         const hta_bf16 *v_cache, const int32_t *cache_lens,
                                         const hta_bf16 *k_spec, const hta_bf16 *v_spec, const uint32_t *mask,
                                         hta_bf16 *o, float *lse, int32_t *dev_err, cudaStream_t stream) {
    if (!dims) return HTA_ERR_INVALID_ARG;
    // hta_workspace_bytes is 0 for invalid dims: let hta_verify report those
    const size_t need = hta_workspace_bytes(dims);
    if (need > (size_t)HTA_NOALLOC_SCRATCH_BYTES) return HTA_ERR_WORKSPACE;
    void *ws = scratch_on_current_device();
    if (!ws) return HTA_ERR_CUDA;
    // the barrier counters at the head of the workspace must start at zero;
    // a previous call that timed out may have left them set
    if (need > 0 && cudaMemsetAsync(ws, 0, 256, stream) != cudaSuccess) return HTA_ERR_CUDA;
    return hta_verify(dims, q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask, o, lse, ws,
                      (size_t)HTA_NOALLOC_SCRATCH_BYTES, dev_err, stream);
}
