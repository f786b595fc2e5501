// CUDA-core (FFMA) attention tile shared by the split-KV kernel (k_cc.cu)
// and the sliding-window kernel (k_window.cu).
//
// Block: 8 warps; a row group holds up to 32 packed query rows, 4 per warp.
// Per 64-key tile: K and V are staged in shared memory (K rows padded so
// 16-byte reads of 8 consecutive rows hit distinct banks), each lane scores
// keys lane and lane+32 against its warp's 4 rows, the warp keeps an online
// softmax in base 2 (scores pre-multiplied by scale*log2 e), and each lane
// accumulates d/32 adjacent output columns.
#pragma once

#include "hta_internal.cuh"

namespace hta {
namespace cct {

constexpr int kTile = 64;
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerGroup = kWarps * kRowsPerWarp;  // 32
constexpr int kThreads = kWarps * 32;

template <int D>
struct CcSmem {
    static constexpr int KST = D + 8;  // padded bf16 row stride of the K tile
    float q[kRowsPerGroup][D];         // scaled queries (scale * log2 e)
    __nv_bfloat16 k[kTile][KST];
    __nv_bfloat16 v[kTile][D];
    float pw[kWarps][kTile][kRowsPerWarp];  // probabilities, [key][row] for float4 broadcast
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
struct RowState {
    float m[kRowsPerWarp];
    float l[kRowsPerWarp];
    float acc[kRowsPerWarp][D / 32];
};

// Loads the scaled queries of the row group into shared memory: row lr maps
// to (t, hq) through row_of(lr, t, hq), which returns false for padding rows.
template <int D, class RowOf>
__device__ __forceinline__ void load_q(const AttnParams &p, CcSmem<D> &sm, int32_t b, RowOf row_of) {
    const int tid = threadIdx.x;
    for (int i = tid; i < kRowsPerGroup * (D / 8); i += kThreads) {
        const int lr = i / (D / 8), c8 = (i % (D / 8)) * 8;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int t = 0, hq = 0;
        if (row_of(lr, t, hq)) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(
                p.q + (((int64_t)b * p.T + t) * p.Hq + hq) * D + c8);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = __bfloat1622float2(h[k]);
                f[2 * k] = x.x * p.scale_log2;
                f[2 * k + 1] = x.y * p.scale_log2;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) sm.q[lr][c8 + k] = f[k];
    }
}

template <int D>
__device__ __forceinline__ void reset(RowState<D> &st) {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        st.m[i] = -INFINITY;
        st.l[i] = 0.f;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) st.acc[i][k] = 0.f;
    }
}

// Scores, visibility, online softmax and O += P V for the staged tile of
// `nvalid` keys. vis(i, jj) says whether row warp*4 + i sees key jj of the
// tile (keys past nvalid are never visible).
template <int D, class Vis>
__device__ __forceinline__ void tile(CcSmem<D> &sm, RowState<D> &st, int nvalid, Vis vis) {
    constexpr int CPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // scores for keys lane, lane+32 against rows warp*4 .. warp*4+3
    float s[kRowsPerWarp][2];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i][0] = s[i][1] = 0.f;
#pragma unroll 4
    for (int c8 = 0; c8 < D; c8 += 8) {
        float kf[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(&sm.k[lane + 32 * h][c8]);
            const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = __bfloat1622float2(hb[k]);
                kf[h][2 * k] = x.x;
                kf[h][2 * k + 1] = x.y;
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const float4 qa = *reinterpret_cast<const float4 *>(&sm.q[warp * kRowsPerWarp + i][c8]);
            const float4 qb = *reinterpret_cast<const float4 *>(&sm.q[warp * kRowsPerWarp + i][c8 + 4]);
            const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                s[i][0] = fmaf(qv[k], kf[0][k], s[i][0]);
                s[i][1] = fmaf(qv[k], kf[1][k], s[i][1]);
            }
        }
    }
    // visibility
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int jj = lane + 32 * h;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
            if (jj >= nvalid || !vis(i, jj)) s[i][h] = -INFINITY;
    }
    // online softmax (base 2)
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const float mx = warp_max(fmaxf(s[i][0], s[i][1]));
        const float m_new = fmaxf(st.m[i], mx);
        float p0 = 0.f, p1 = 0.f, alpha = 1.f;
        if (m_new > -INFINITY) {
            alpha = exp2f(st.m[i] - m_new);  // 0 when the old max is -inf
            p0 = exp2f(s[i][0] - m_new);
            p1 = exp2f(s[i][1] - m_new);
            st.m[i] = m_new;
        }
        st.l[i] = st.l[i] * alpha + warp_sum(p0 + p1);
#pragma unroll
        for (int k = 0; k < CPL; ++k) st.acc[i][k] *= alpha;
        sm.pw[warp][lane][i] = p0;
        sm.pw[warp][lane + 32][i] = p1;
    }
    __syncwarp();
    // O += P V
#pragma unroll 4
    for (int jj = 0; jj < kTile; ++jj) {
        const float4 pj = *reinterpret_cast<const float4 *>(&sm.pw[warp][jj][0]);
        float vf[CPL];
        if constexpr (CPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(&sm.v[jj][lane * 4]);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
            const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
            vf[0] = a.x; vf[1] = a.y; vf[2] = c.x; vf[3] = c.y;
        } else {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&sm.v[jj][lane * 2]));
            vf[0] = a.x; vf[1] = a.y;
        }
        const float pv[4] = {pj.x, pj.y, pj.z, pj.w};
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
            for (int k = 0; k < CPL; ++k) st.acc[i][k] = fmaf(pv[i], vf[k], st.acc[i][k]);
    }
    __syncwarp();
}

}  // namespace cct
}  // namespace hta
