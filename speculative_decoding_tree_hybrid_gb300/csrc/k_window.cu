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
// A draft step has few queries (often one per sequence: 4 packed rows per KV
// head with GQA), so the CTA splits the keys, not the rows: one CTA per
// (sequence, KV head, group of 4 packed rows). The group's visible positions
// are walked in 64-key tiles; one thread copies each tile's K and V rows from
// the ring into shared memory with bulk copies (two when the tile wraps past
// the ring's end), into a ring of three stages so two tiles are in flight
// while the current one is used. Warp w takes keys 8w .. 8w+7 of every tile: its lanes
// split the head dimension (d/32 columns each), a dot product is a warp
// reduction, and the same columns then accumulate P V with no exchange.
// Each warp keeps an online softmax (base 2) per row; the 8 partial states
// are merged in shared memory by the log-sum-exp rule at the end.
#include "hta_internal.cuh"
#include "hta_launch.h"
#include "tc_ptx.cuh"

namespace hta {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 4;               // packed query rows per CTA
constexpr int kTile = 64;              // keys per tile
constexpr int kKeysPerWarp = kTile / kWarps;
constexpr int kStages = 3;

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
struct WinMerge {
    float acc[kWarps][kRows][D];  // per-warp unnormalised outputs
    float m[kWarps][kRows], l[kWarps][kRows];
};

template <int D>
struct WinSmem {
    union {
        struct {
            __nv_bfloat16 k[kStages][kTile][D];  // stages of key rows
            __nv_bfloat16 v[kStages][kTile][D];
        } ring;
        WinMerge<D> merge;  // reuses the idle ring after the last tile
    };
    uint64_t full[kStages];
    int32_t status;
};

template <int D>
__global__ void __launch_bounds__(kThreads)
    k_window_attn(const __grid_constant__ AttnParams p, const int32_t *__restrict__ pos, int32_t W, int32_t S,
                  int32_t n_rg) {
    constexpr int CPL = D / 32;  // columns per lane
    extern __shared__ __align__(128) unsigned char smem_raw[];
    WinSmem<D> &sm = *reinterpret_cast<WinSmem<D> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t rg = blockIdx.x % n_rg;
    const int32_t kvh = (blockIdx.x / n_rg) % p.Hkv;
    const int32_t b = blockIdx.x / (n_rg * p.Hkv);
    const int32_t R = p.T * p.G;  // packed rows of this KV head
    const int32_t r_base = rg * kRows;
    const int32_t nrows = min(kRows, R - r_base);
    int64_t P = pos[b];
    if (P < 0) {
        if (kvh == 0 && rg == 0 && threadIdx.x == 0) flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
        P = 0;
    }
    // positions any row of the group sees: [j_begin, j_end)
    const int64_t j_begin = max((int64_t)0, P + r_base / p.G - W + 1);
    const int64_t j_end = P + (r_base + nrows - 1) / p.G + 1;
    const int n_tiles = (int)((j_end - j_begin + kTile - 1) / kTile);
    const int64_t kv_off = ((int64_t)b * p.Hkv + kvh) * S;

    // tile i: positions j_begin + 64 i .. (< j_end) into stage i % 2, as one or
    // two contiguous runs of ring slots
    auto issue = [&](int i) {
        const int64_t j0 = j_begin + (int64_t)i * kTile;
        const int n = (int)min((int64_t)kTile, j_end - j0);
        const int64_t s0 = j0 % S;
        const int n1 = (int)min((int64_t)n, S - s0);  // rows before the wrap
        const uint32_t bar = tc::smem_u32(&sm.full[i % kStages]);
        const uint32_t row = D * 2;
        tc::mbar_arrive_expect_tx(bar, (uint32_t)n * row * 2);
        tc::bulk_load(tc::smem_u32(&sm.ring.k[i % kStages][0][0]), p.k_cache + (kv_off + s0) * D, (uint32_t)n1 * row, bar);
        tc::bulk_load(tc::smem_u32(&sm.ring.v[i % kStages][0][0]), p.v_cache + (kv_off + s0) * D, (uint32_t)n1 * row, bar);
        if (n1 < n) {
            tc::bulk_load(tc::smem_u32(&sm.ring.k[i % kStages][n1][0]), p.k_cache + kv_off * D, (uint32_t)(n - n1) * row, bar);
            tc::bulk_load(tc::smem_u32(&sm.ring.v[i % kStages][n1][0]), p.v_cache + kv_off * D, (uint32_t)(n - n1) * row, bar);
        }
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) tc::mbar_init(tc::smem_u32(&sm.full[st]), 1);
        tc::mbar_fence_init();
        sm.status = 1;
        for (int i = 0; i < kStages - 1 && i < n_tiles; ++i) issue(i);
    }

    // this lane's columns of the group's queries, scaled; padding rows are zero
    float q[kRows][CPL];
    int64_t tq[kRows];  // query position of each row (-1: padding, sees nothing)
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        tq[i] = -1;
#pragma unroll
        for (int c = 0; c < CPL; ++c) q[i][c] = 0.f;
        if (i < nrows) {
            const int r = r_base + i, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
            tq[i] = P + t;
            const __nv_bfloat16 *qr = p.q + (((int64_t)b * p.T + t) * p.Hq + hq) * D + lane * CPL;
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qr + c));
                q[i][c] = x.x * p.scale_log2;
                q[i][c + 1] = x.y * p.scale_log2;
            }
        }
    }
    float m[kRows], l[kRows], acc[kRows][CPL];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[i][c] = 0.f;
    }
    __syncthreads();  // barriers initialised

    for (int it = 0; it < n_tiles; ++it) {
        // tile it + 2 goes to the stage that tile it - 1 released at the end of the last iteration
        if (threadIdx.x == 0 && it + kStages - 1 < n_tiles) issue(it + kStages - 1);
        if (threadIdx.x == 0) {
            const uint64_t t0 = cycles_now();
            while (!tc::mbar_try_wait(tc::smem_u32(&sm.full[it % kStages]), (it / kStages) & 1)) {
                if (cycles_now() - t0 > kWaitLimitCycles) {
                    flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                    sm.status = 0;
                    break;
                }
            }
        }
        __syncthreads();
        if (!sm.status) break;
        const int64_t j0 = j_begin + (int64_t)it * kTile;
        const int n = (int)min((int64_t)kTile, j_end - j0);
        const int k_lo = warp * kKeysPerWarp, k_hi = min(n, k_lo + kKeysPerWarp);
        // scores of this warp's keys (lanes over the columns, then a warp sum)
        float s[kRows][kKeysPerWarp];
#pragma unroll
        for (int kk = 0; kk < kKeysPerWarp; ++kk) {
            const int key = k_lo + kk;
            float kf[CPL];
            if (key < k_hi) {
#pragma unroll
                for (int c = 0; c < CPL; c += 2) {
                    const float2 x = __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162 *>(&sm.ring.k[it % kStages][key][lane * CPL + c]));
                    kf[c] = x.x;
                    kf[c + 1] = x.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c) kf[c] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                float d = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) d = fmaf(q[i][c], kf[c], d);
                s[i][kk] = d;
            }
        }
#pragma unroll
        for (int kk = 0; kk < kKeysPerWarp; ++kk)
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const int64_t j = j0 + k_lo + kk;
                const float d = wsum(s[i][kk]);
                // visibility: P + t - W < j <= P + t, and a key of this tile
                s[i][kk] = (k_lo + kk < k_hi && j <= tq[i] && j > tq[i] - W) ? d : -INFINITY;
            }
        // online softmax per row over the warp's keys, then O += P V
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < kKeysPerWarp; ++kk) mx = fmaxf(mx, s[i][kk]);
            const float m_new = fmaxf(m[i], mx);
            if (m_new > -INFINITY) {
                const float alpha = exp2f(m[i] - m_new);  // 0 while the old max is -inf
                l[i] *= alpha;
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc[i][c] *= alpha;
                m[i] = m_new;
#pragma unroll
                for (int kk = 0; kk < kKeysPerWarp; ++kk) {
                    const float pk = exp2f(s[i][kk] - m_new);  // 0 for an invisible key
                    s[i][kk] = pk;
                    l[i] += pk;
                }
            }
        }
#pragma unroll
        for (int kk = 0; kk < kKeysPerWarp; ++kk) {
            const int key = k_lo + kk;
            if (key >= k_hi) break;  // rows past the copied ones are stale
            float vf[CPL];
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162 *>(&sm.ring.v[it % kStages][key][lane * CPL + c]));
                vf[c] = x.x;
                vf[c + 1] = x.y;
            }
#pragma unroll
            for (int i = 0; i < kRows; ++i)
                if (m[i] > -INFINITY) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) acc[i][c] = fmaf(s[i][kk], vf[c], acc[i][c]);
                }
        }
        __syncthreads();  // stage it % kStages is free for tile it + kStages
    }

    // merge the warps' partial softmaxes
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) sm.merge.acc[warp][i][lane * CPL + c] = acc[i][c];
        if (lane == 0) {
            sm.merge.m[warp][i] = m[i];
            sm.merge.l[warp][i] = l[i];
        }
    }
    __syncthreads();
    const bool ok = sm.status != 0;
    for (int x = threadIdx.x; x < nrows * D; x += kThreads) {
        const int i = x / D, c = x % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.merge.m[w][i]);
        float num = 0.f, den = 0.f;
        if (M > -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float e = exp2f(sm.merge.m[w][i] - M);  // 0 for a warp that saw no key
                num = fmaf(e, sm.merge.acc[w][i][c], num);
                den = fmaf(e, sm.merge.l[w][i], den);
            }
        }
        const int r = r_base + i, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
        const int64_t out_row = ((int64_t)b * p.T + t) * p.Hq + hq;
        const float nan = __int_as_float(0x7fc00000);  // a timed-out copy leaves NaN outputs
        ((__nv_bfloat16 *)p.out_o)[out_row * D + c] = __float2bfloat16_rn(!ok ? nan : den > 0.f ? num / den : 0.f);
        if (c == 0) p.out_lse[out_row] = !ok ? nan : den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
}

template <int D>
cudaError_t window_launch_t(const AttnParams &p, const int32_t *pos, int32_t W, int32_t S, cudaStream_t stream) {
    const int32_t n_rg = (p.T * p.G + kRows - 1) / kRows;
    const int64_t grid = (int64_t)p.B * p.Hkv * n_rg;
    if (grid <= 0 || grid > 0x7fffffff) return cudaErrorInvalidValue;
    const size_t smem = sizeof(WinSmem<D>);
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
