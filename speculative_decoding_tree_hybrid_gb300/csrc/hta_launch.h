// Host-side launch interface between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>

#include "hta_internal.cuh"

namespace hta {

// The attention kernels merge their split-KV partials after a grid-wide
// barrier, so every CTA of the grid must be resident at once. Their grids are
// sized by the occupancy query to fit the device, and none of them lets a
// dependent start before it has finished (no early launch_dependents: with
// clusters of three CTAs that measured as a stall), so nothing launched after
// a grid can hold SMs it needs; they are launched as ordinary grids by
// default, 2.2 us per call sooner back to back than cooperative ones.
// HTA_COOPERATIVE=1 (read on every call) asks for a cooperative launch, which
// also guarantees co-residency against work on other streams.
inline bool cooperative_requested() {
    const char *s = getenv("HTA_COOPERATIVE");
    return s && s[0] == '1' && s[1] == 0;
}

// Launches `kern` with the n attributes in attrs[0 .. n) plus programmatic
// stream serialization (attrs must have room for n + 1): the kernel may then
// start while the kernel before it on the stream is still running, and waits
// for it (griddep_wait) before reading what that kernel writes. The mask
// build is the only kernel here that lets its dependent start early, and only
// once every kernel before it has finished, so the attention kernels wait
// only before reading the mask. If the runtime rejects that
// attribute with the others, the launch is repeated without it, and so are
// all later launches of the process.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(cudaLaunchConfig_t cfg, cudaLaunchAttribute *attrs, int n, void (*kern)(KArgs...),
                             Args &&...args) {
    static std::atomic<int> allowed{1};
    cfg.attrs = attrs;
    if (allowed.load(std::memory_order_relaxed)) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = (unsigned)(n + 1);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
        if (e == cudaSuccess) return e;
        (void)cudaGetLastError();
        allowed.store(0, std::memory_order_relaxed);
    }
    cfg.numAttrs = (unsigned)n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// CUDA-core path (k_cc.cu)
int cc_rows_per_group();
int cc_tile();
int cc_max_grid(int d, int B, int num_sms);
cudaError_t cc_launch(const AttnParams &p, bool direct, int grid, cudaStream_t stream);

// tcgen05 path (k_tc.cu)
int tc_rows_per_group();
int tc_tile();
int tc_max_grid(int B, int num_sms);
cudaError_t tc_launch(const AttnParams &p, int grid, cudaStream_t stream);

// clustered tcgen05 path, clusters of 2 to 4 CTAs sharing every K/V tile (k_tc2.cu)
int tc2_tile();
int tc2_rows_per_sub();
int tc2_max_grid(int B, int num_sms, int csize);
cudaError_t tc2_launch(const AttnParams &p, int grid, cudaStream_t stream);

// accept walk and KV commit (k_accept.cu); `st` is the cache storage (all
// zero: contiguous head-major)
struct KvStore {
    int32_t nhd, page_size, max_pages, num_pages;
    const int32_t *block_table;
};
cudaError_t accept_launch(const int32_t *parents, const int32_t *draft, const int32_t *target, int B, int T,
                          int Hkv, int d, int64_t Lmax, const void *k_spec, const void *v_spec, void *k_cache,
                          void *v_cache, int32_t *cache_lens, int32_t *accepted, int32_t *n_accepted,
                          int32_t *next_token, int32_t *dev_err, const KvStore &st, cudaStream_t stream);

// draft-model sliding-window (W) self-attention over a ring of S slots (k_window.cu)
cudaError_t window_launch(const AttnParams &p, const int32_t *pos, int32_t W, int32_t S, cudaStream_t stream);

// LogitSpec draft-tree builder (k_lspec.cu)
struct LspecParams {
    const float *logits;       // [B][V]
    const int32_t *hist;       // [B][Lh_max]
    const int32_t *hist_len;   // [B]
    int32_t *parents, *tokens;  // [B][T]
    int32_t *n_nodes, *next_token;  // [B]
    int32_t *dev_err;
    int64_t Lh_max;
    int32_t B, V, T, k, m;
    int32_t keep[HTA_LSPEC_KMAX + 1];
};
cudaError_t lspec_launch(const LspecParams &p, cudaStream_t stream);

// tree mask (k_mask.cu)
cudaError_t mask_launch(const int32_t *parents, int B, int T, uint32_t *mask, int32_t *dev_err,
                        cudaStream_t stream);

// two-part merge (k_merge.cu)
cudaError_t merge2_launch(int64_t rows, int d, const float *o_c, const float *lse_c, const float *o_s,
                          const float *lse_s, __nv_bfloat16 *o, float *lse, cudaStream_t stream);

}  // namespace hta
