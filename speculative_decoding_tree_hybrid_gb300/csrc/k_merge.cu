// Stand-alone log-sum-exp merge of the cached part and the speculative part
// ("LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", Korean summary section 2.C "aggregation"; Dutch
// summary Methodologie section 3, last bullet):
//   m = max(lse_c, lse_s), w_c = e^(lse_c - m), w_s = e^(lse_s - m),
//   o = (w_c o_c + w_s o_s) / (w_c + w_s), lse = m + ln(w_c + w_s).
// A part whose lse is -inf weighs zero; both -inf gives o = 0, lse = -inf.
// One warp per (b, t, hq) row; lanes own d/32 adjacent columns.
#include "hta_launch.h"

namespace hta {
namespace {

template <int D>
__global__ void __launch_bounds__(256) k_merge2(int64_t rows, const float *__restrict__ o_c,
                                                const float *__restrict__ lse_c,
                                                const float *__restrict__ o_s,
                                                const float *__restrict__ lse_s,
                                                __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
    constexpr int CPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float a = lse_c[row], b = lse_s[row];
    const float m = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, out_lse = -INFINITY;
    if (m > -INFINITY) {
        wa = __expf(a - m);
        wb = __expf(b - m);
        out_lse = m + __logf(wa + wb);
    }
    const float inv = (wa + wb) > 0.f ? 1.f / (wa + wb) : 0.f;
    const float *pc = o_c + row * D + lane * CPL;
    const float *ps = o_s + row * D + lane * CPL;
    __nv_bfloat16 *po = o + row * D + lane * CPL;
#pragma unroll
    for (int k = 0; k < CPL; k += 2) {
        const float x0 = wa > 0.f ? wa * pc[k] : 0.f, x1 = wa > 0.f ? wa * pc[k + 1] : 0.f;
        const float y0 = wb > 0.f ? wb * ps[k] : 0.f, y1 = wb > 0.f ? wb * ps[k + 1] : 0.f;
        *reinterpret_cast<__nv_bfloat162 *>(po + k) =
            __floats2bfloat162_rn((x0 + y0) * inv, (x1 + y1) * inv);
    }
    if (lane == 0) lse[row] = out_lse;
}

}  // namespace

cudaError_t merge2_launch(int64_t rows, int d, const float *o_c, const float *lse_c, const float *o_s,
                          const float *lse_s, __nv_bfloat16 *o, float *lse, cudaStream_t stream) {
    const int64_t blocks = (rows + 7) / 8;
    if (d == 128)
        k_merge2<128><<<(unsigned)blocks, 256, 0, stream>>>(rows, o_c, lse_c, o_s, lse_s, o, lse);
    else
        k_merge2<64><<<(unsigned)blocks, 256, 0, stream>>>(rows, o_c, lse_c, o_s, lse_s, o, lse);
    return cudaGetLastError();
}

}  // namespace hta
