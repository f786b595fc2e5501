// Sliding-window self-attention of the draft model ("LongSpec: Long-Context
// Lossless Speculative Decoding with Efficient Drafting and Verification",
// Korean summary section 2.A "memory-efficient architecture"; Dutch summary
// Methodologie section 1, "Self-Attention"): each query attends causally to
// the W most recent positions up to and including its own (W = 512 in the
// pages), so the draft model's own KV cache keeps a fixed size whatever the
// context length.
//
// Ring layout: position j of sequence b lives in slot j mod S of
// k_ring/v_ring [B][Hkv][S][d]. The T queries of a call sit at positions
// P_b .. P_b + T - 1 (their keys are already in the ring); query t sees
// positions j with P_b + t - W < j <= P_b + t and j >= 0, so the ring needs
// S >= W + T - 1 slots (the first query still reads W - 1 older positions).
//
// One CTA per (sequence, KV head, group of 32 packed query rows); the group's
// visible positions span at most W + T - 1 keys, walked in 64-key tiles with
// the CUDA-core tile of cc_tile.cuh, and the CTA writes the normalised output
// directly (no split, no workspace).
#include "cc_tile.cuh"
#include "hta_internal.cuh"
#include "hta_launch.h"

namespace hta {
namespace {

using cct::CcSmem;
using cct::kRowsPerGroup;
using cct::kRowsPerWarp;
using cct::kThreads;
using cct::kTile;
using cct::RowState;

template <int D>
__global__ void __launch_bounds__(kThreads)
    k_window_attn(const __grid_constant__ AttnParams p, const int32_t *__restrict__ pos, int32_t W, int32_t S,
                  int32_t n_rg) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    CcSmem<D> &sm = *reinterpret_cast<CcSmem<D> *>(smem_raw);
    RowState<D> st;
    constexpr int CPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t rg = blockIdx.x % n_rg;
    const int32_t kvh = (blockIdx.x / n_rg) % p.Hkv;
    const int32_t b = blockIdx.x / (n_rg * p.Hkv);
    const int32_t R = p.T * p.G;  // packed rows of this KV head
    const int32_t r_base = rg * kRowsPerGroup;
    const int32_t nrows = min(kRowsPerGroup, R - r_base);
    int32_t P = pos[b];
    if (P < 0) {
        if (kvh == 0 && rg == 0 && threadIdx.x == 0) flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
        P = 0;
    }

    cct::load_q<D>(p, sm, b, [&](int lr, int &t, int &hq) {
        if (lr >= nrows) return false;
        const int r = r_base + lr;
        t = r / p.G;
        hq = kvh * p.G + (r - t * p.G);
        return true;
    });
    cct::reset<D>(st);

    // positions any row of the group sees: [j_begin, j_end)
    const int32_t t_lo = r_base / p.G, t_hi = (r_base + nrows - 1) / p.G;
    const int64_t j_begin = max((int64_t)0, (int64_t)P + t_lo - W + 1);
    const int64_t j_end = (int64_t)P + t_hi + 1;
    const int64_t kv_off = ((int64_t)b * p.Hkv + kvh) * S;
    for (int64_t j0 = j_begin; j0 < j_end; j0 += kTile) {
        const int nvalid = (int)min((int64_t)kTile, j_end - j0);
        __syncthreads();  // previous tile fully consumed (and the queries written)
        for (int i = threadIdx.x; i < kTile * (D / 8); i += kThreads) {
            const int jj = i / (D / 8), c8 = (i % (D / 8)) * 8;
            uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
            if (jj < nvalid) {
                const int64_t slot = (j0 + jj) % S;
                kr = __ldg(reinterpret_cast<const uint4 *>(p.k_cache + (kv_off + slot) * D + c8));
                vr = __ldg(reinterpret_cast<const uint4 *>(p.v_cache + (kv_off + slot) * D + c8));
            }
            *reinterpret_cast<uint4 *>(&sm.k[jj][c8]) = kr;
            *reinterpret_cast<uint4 *>(&sm.v[jj][c8]) = vr;
        }
        __syncthreads();
        cct::tile<D>(sm, st, nvalid, [&](int i, int jj) {
            const int lr = warp * kRowsPerWarp + i;
            if (lr >= nrows) return false;
            const int64_t t = (r_base + lr) / p.G, j = j0 + jj;
            return j <= P + t && j > P + t - W;
        });
    }

    // normalised output: every real row sees at least its own position
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int lr = warp * kRowsPerWarp + i;
        if (lr >= nrows) continue;
        const int r = r_base + lr, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
        const int64_t out_row = ((int64_t)b * p.T + t) * p.Hq + hq;
        const bool any = st.l[i] > 0.f;
        const float inv = any ? 1.f / st.l[i] : 0.f;
        const float lse = any ? (st.m[i] + log2f(st.l[i])) * kLn2 : -INFINITY;
        __nv_bfloat16 *o = (__nv_bfloat16 *)p.out_o + out_row * D + lane * CPL;
#pragma unroll
        for (int k = 0; k < CPL; k += 2)
            *reinterpret_cast<__nv_bfloat162 *>(o + k) =
                __floats2bfloat162_rn(st.acc[i][k] * inv, st.acc[i][k + 1] * inv);
        if (lane == 0) p.out_lse[out_row] = lse;
    }
}

template <int D>
cudaError_t window_launch_t(const AttnParams &p, const int32_t *pos, int32_t W, int32_t S, cudaStream_t stream) {
    const int32_t n_rg = (p.T * p.G + kRowsPerGroup - 1) / kRowsPerGroup;
    const int64_t grid = (int64_t)p.B * p.Hkv * n_rg;
    if (grid <= 0 || grid > 0x7fffffff) return cudaErrorInvalidValue;
    const size_t smem = sizeof(CcSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(k_window_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_window_attn<D><<<(unsigned)grid, kThreads, smem, stream>>>(p, pos, W, S, n_rg);
    return cudaGetLastError();
}

}  // namespace

cudaError_t window_launch(const AttnParams &p, const int32_t *pos, int32_t W, int32_t S, cudaStream_t stream) {
    return p.d == 128 ? window_launch_t<128>(p, pos, W, S, stream) : window_launch_t<64>(p, pos, W, S, stream);
}

}  // namespace hta
