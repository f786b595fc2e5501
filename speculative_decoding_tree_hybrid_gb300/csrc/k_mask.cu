// Tree mask builder: parents -> bit-packed ancestor-or-self mask.
//
// The draft tree ("LogitSpec: Accelerating Retrieval-based Speculative
// Decoding via Next Next Token Speculation", section 2, workflow step 2) is
// verified branch-parallel under a tree attention mask; node i may see tree
// token j iff j is i or one of i's ancestors.
//
// One CTA per tree, one thread per node. Pointer jumping: after round k the
// row of node i holds the 2^k nearest nodes of its root path and jump[i] is its
// 2^k-th ancestor (-1 past the root); rows merge as
//   row_{k+1}(i) = row_k(i) | row_k(jump_k(i)),  jump_{k+1}(i) = jump_k(jump_k(i)),
// so ceil(log2 T) + 1 rounds cover every path of a tree of T <= 256 nodes.
// Parents outside [-1, i-1] mark the tree invalid: its rows are written as
// zero and HTA_DEVERR_BAD_TREE is raised.
#include "hta_launch.h"

namespace hta {
namespace {

constexpr int kMaxW = HTA_TMAX / 32;

__global__ void __launch_bounds__(HTA_TMAX) k_build_mask(const int32_t *__restrict__ parents, int T,
                                                        int W, uint32_t *__restrict__ mask,
                                                        int32_t *dev_err) {
    __shared__ uint32_t rows[2][HTA_TMAX][kMaxW];
    __shared__ int32_t jump[2][HTA_TMAX];
    __shared__ int bad_s;
    const int b = blockIdx.x, i = threadIdx.x;
    const int32_t *par = parents + (int64_t)b * T;
    // launched as a programmatic dependent: the kernel before it (often the
    // attention of the previous step, which reads the mask) has finished and
    // its memory is visible from here on
    tc::griddep_wait();
    // only now may the attention launch start: every kernel before this one
    // has finished, so the attention waits for nothing but this mask
    tc::griddep_launch_dependents();
    if (i == 0) bad_s = 0;
    __syncthreads();
    int32_t pi = -1;
    if (i < T) {
        pi = par[i];
        if (pi < -1 || pi >= i) bad_s = 1;  // benign race: every writer stores 1
        for (int w = 0; w < W; ++w) rows[0][i][w] = (w == (i >> 5)) ? (1u << (i & 31)) : 0u;
        jump[0][i] = pi;
    }
    __syncthreads();
    const bool bad = bad_s != 0;
    int cur = 0;
    if (!bad) {
        for (int span = 1; span < 2 * T; span <<= 1) {
            if (i < T) {
                const int32_t j = jump[cur][i];
                for (int w = 0; w < W; ++w)
                    rows[cur ^ 1][i][w] = rows[cur][i][w] | (j >= 0 ? rows[cur][j][w] : 0u);
                jump[cur ^ 1][i] = j >= 0 ? jump[cur][j] : -1;
            }
            __syncthreads();
            cur ^= 1;
        }
    }
    if (i < T) {
        uint32_t *out = mask + ((int64_t)b * T + i) * W;
        for (int w = 0; w < W; ++w) out[w] = bad ? 0u : rows[cur][i][w];
    }
    if (bad && i == 0) flag_error(dev_err, HTA_DEVERR_BAD_TREE);
}

}  // namespace

cudaError_t mask_launch(const int32_t *parents, int B, int T, uint32_t *mask, int32_t *dev_err,
                        cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(((T + 31) / 32) * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    return launch_dependent(cfg, attr, 0, k_build_mask, parents, T, (T + 31) / 32, mask, dev_err);
}

}  // namespace hta
