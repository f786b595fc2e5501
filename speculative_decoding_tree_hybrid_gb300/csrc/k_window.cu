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
// are walked in 64-key tiles; a copy warp moves each tile's K and V rows from
// the ring into shared memory with bulk copies (two when the tile wraps past
// the ring's end), into a ring of three stages, refilling a stage as soon as
// all eight compute warps have released it (full and empty barriers per
// stage, no block-wide barrier per tile). Warp w takes keys 8w .. 8w+7 of
// every tile: its lanes split the head dimension (d/32 columns each) for the
// 32 (key, row) dot products, each lane holding pair p in slot p ^ lane, so
// that a butterfly reduce-scatter of 31 shuffles and adds (the kept half is
// always the low one: no selects) leaves lane L the full score of key L / 4
// and row L % 4; the softmax of a row runs over its 8
// lanes (one exponential per lane), and the probabilities go back to every
// lane through shared memory for P V, accumulated on the same columns.
// Each warp keeps an online softmax (base 2) per row; the 8 partial states
// are merged in shared memory by the log-sum-exp rule at the end. The dot
// products (two rows per instruction), the rescale and P V (two columns per
// instruction) run on Blackwell's packed fp32 pairs.
#include "hta_internal.cuh"
#include "hta_launch.h"
#include "tc_ptx.cuh"

namespace hta {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = (kWarps + 1) * 32;  // compute warps and one copy warp
constexpr int kRows = 4;               // packed query rows per CTA
constexpr int kTile = 64;              // keys per tile
constexpr int kKeysPerWarp = kTile / kWarps;
constexpr int kStages = 3;

// max / sum over the 8 lanes that share lane % 4
__device__ __forceinline__ float row_max(float v) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One step of the reduce-scatter when lane L holds pair p in slot p ^ L:
// the pairs a lane keeps at step n are in slots [0, n), the ones it hands
// to lane L ^ n in [n, 2n), where that lane keeps the same pairs in [0, n).
template <int n>
__device__ __forceinline__ void fold_step(float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < n; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q + n], n);
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
    alignas(16) float prob[kWarps][32];  // a warp's probabilities of one tile, (key, row) pair L = 4 key + row
    uint64_t full[kStages];
    uint64_t empty[kStages];  // kWarps arrivals: every compute warp is done with the stage
    int32_t status;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
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
        for (int st = 0; st < kStages; ++st) {
            tc::mbar_init(tc::smem_u32(&sm.full[st]), 1);
            tc::mbar_init(tc::smem_u32(&sm.empty[st]), kWarps);
        }
        tc::mbar_fence_init();
        sm.status = 1;
    }

    // this lane's columns of the group's queries, scaled; padding rows are zero
    float q[kRows][CPL];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) q[i][c] = 0.f;
        const int ir = i ^ (lane & 3);  // slot i of this lane holds row i ^ (lane % 4)
        if (ir < nrows) {
            const int r = r_base + ir, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
            const __nv_bfloat16 *qr = p.q + (((int64_t)b * p.T + t) * p.Hq + hq) * D + lane * CPL;
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(qr + c));
                q[i][c] = x.x * p.scale_log2;
                q[i][c + 1] = x.y * p.scale_log2;
            }
        }
    }
    // running max and denominator of row lane % 4 (the 8 lanes of a row hold
    // the same values); O of every row on this lane's columns
    const int row_l = lane & 3, key_l = lane >> 2;
    const int64_t tq_l = row_l < nrows ? P + (r_base + row_l) / p.G : -1;
    float m_l = -INFINITY, l_l = 0.f, acc[kRows][CPL];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[i][c] = 0.f;
    __syncthreads();  // barriers initialised

    volatile int32_t *status = &sm.status;
    int n_issued = 0;  // copy warp, lane 0: tiles whose copies were issued
    if (warp == kWarps) {
        // the copy warp: tile i goes to stage i % kStages once every compute
        // warp has released tile i - kStages
        if (lane == 0) {
            for (int i = 0; i < n_tiles && *status; ++i) {
                if (i >= kStages) {
                    const uint64_t t0 = cycles_now();
                    bool got = true;
                    while (!tc::mbar_try_wait(tc::smem_u32(&sm.empty[i % kStages]), (i / kStages - 1) & 1)) {
                        if (!*status) {
                            got = false;
                            break;
                        }
                        if (cycles_now() - t0 > kWaitLimitCycles) {
                            flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                            *status = 0;
                            got = false;
                            break;
                        }
                    }
                    if (!got) break;
                }
                issue(i);
                n_issued = i + 1;
            }
        }
    } else {
    for (int it = 0; it < n_tiles; ++it) {
        bool got = true;
        {
            const uint64_t t0 = cycles_now();
            while (!tc::mbar_try_wait(tc::smem_u32(&sm.full[it % kStages]), (it / kStages) & 1)) {
                if (!*status || cycles_now() - t0 > kWaitLimitCycles) {
                    got = false;
                    break;
                }
            }
        }
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0 && *status) {
                flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                *status = 0;
            }
            break;
        }
        const int64_t j0 = j_begin + (int64_t)it * kTile;
        const int n = (int)min((int64_t)kTile, j_end - j0);
        const int k_lo = warp * kKeysPerWarp, k_hi = min(n, k_lo + kKeysPerWarp);
        // partial scores of this warp's (key, row) pairs on this lane's columns
        float v[32];
#pragma unroll
        for (int kk = 0; kk < kKeysPerWarp; ++kk) {
            const int key = k_lo + (kk ^ (lane >> 2));  // slot kk of this lane: key kk ^ (lane / 4)
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
            // rows (0, 1) and (2, 3) in pairs, columns in order
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                tc::fma2v(d0, d1, q[0][c], q[1][c], kf[c], kf[c]);
                tc::fma2v(d2, d3, q[2][c], q[3][c], kf[c], kf[c]);
            }
            v[kk * kRows + 0] = d0;
            v[kk * kRows + 1] = d1;
            v[kk * kRows + 2] = d2;
            v[kk * kRows + 3] = d3;
        }
        fold_step<16>(v);
        fold_step<8>(v);
        fold_step<4>(v);
        fold_step<2>(v);
        fold_step<1>(v);
        // lane L: key k_lo + L / 4, row L % 4; visible when P + t - W < j <= P + t
        const int64_t j = j0 + k_lo + key_l;
        const float s = (k_lo + key_l < k_hi && j <= tq_l && j > tq_l - W) ? v[0] : -INFINITY;
        // online softmax of each row over its 8 lanes
        const float m_new = fmaxf(m_l, row_max(s));
        float alpha = 1.f, pr = 0.f;
        if (m_new > -INFINITY) {
            alpha = exp2f(m_l - m_new);  // 0 while the old max is -inf
            pr = exp2f(s - m_new);       // 0 for an invisible key
            m_l = m_new;
        }
        l_l = l_l * alpha + row_sum(pr);
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const float a = __shfl_sync(0xffffffffu, alpha, i);  // lane i holds row i
#pragma unroll
            for (int c = 0; c < CPL; c += 2) tc::mul2s(acc[i][c], acc[i][c + 1], a);
        }
        sm.prob[warp][lane] = pr;
        __syncwarp();
        // O += P V on this lane's columns
#pragma unroll
        for (int kk = 0; kk < kKeysPerWarp; ++kk) {
            const int key = k_lo + kk;
            if (key >= k_hi) break;  // rows past the copied ones are stale
            const float4 pk = *reinterpret_cast<const float4 *>(&sm.prob[warp][kk * kRows]);
            float vf[CPL];
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 x = __bfloat1622float2(
                    *reinterpret_cast<const __nv_bfloat162 *>(&sm.ring.v[it % kStages][key][lane * CPL + c]));
                vf[c] = x.x;
                vf[c + 1] = x.y;
            }
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                tc::fma2v(acc[0][c], acc[0][c + 1], pk.x, pk.x, vf[c], vf[c + 1]);
                tc::fma2v(acc[1][c], acc[1][c + 1], pk.y, pk.y, vf[c], vf[c + 1]);
                tc::fma2v(acc[2][c], acc[2][c + 1], pk.z, pk.z, vf[c], vf[c + 1]);
                tc::fma2v(acc[3][c], acc[3][c + 1], pk.w, pk.w, vf[c], vf[c + 1]);
            }
        }
        __syncwarp();  // prob is rewritten by the next tile
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sm.empty[it % kStages]));  // this warp is done with the stage
    }
    }
    __syncthreads();  // every warp is done with the ring, which the merge reuses
    if (!*status) {  // the same in every thread from here on
        // a wait gave up: copies may still be landing in the ring. Wait
        // (bounded) for the latest tile of each stage, whose phase is the only
        // one that can still be open.
        if (warp == kWarps && lane == 0) {
            for (int i = max(0, n_issued - kStages); i < n_issued; ++i) {
                const uint64_t t0 = cycles_now();
                while (!tc::mbar_try_wait(tc::smem_u32(&sm.full[i % kStages]), (i / kStages) & 1))
                    if (cycles_now() - t0 > kWaitLimitCycles) break;
            }
        }
        __syncthreads();
    }

    // merge the warps' partial softmaxes
    if (warp < kWarps) {
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) sm.merge.acc[warp][i][lane * CPL + c] = acc[i][c];
        }
        if (lane < kRows) {  // lane i holds row i
            sm.merge.m[warp][lane] = m_l;
            sm.merge.l[warp][lane] = l_l;
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
