// Internal definitions shared by the libhta kernels: launch parameters, the
// static split-KV schedule, the grid barrier and the cross-split /
// cross-part log-sum-exp merge.
//
// Work decomposition (both kernel paths):
//   segment s = ((b * Hkv) + kvh) * n_rg + rg : one KV head of one sequence and
//               one group of its packed query rows (packed row r = t*G + g, so
//               all G query heads of a KV head share every K/V tile);
//   unit      = one tile of `tile` keys: tree tiles first (masked), then the
//               cache tiles of that segment (unmasked, keys j < L_b);
//   CTA c of the persistent grid owns units [c*U/grid, (c+1)*U/grid) of the
//   linearised unit space, so every CTA gets the same number of tiles
//   whatever the mix of cache lengths; a CTA whose range crosses a segment
//   boundary emits one partial per segment piece.
//   Piece (s, c) writes its partial, one record per query row
//   [un-normalised O (d floats) | running max m (log2 units) | denominator l |
//   2 pad], to slot s + c; a monotone staircase of pieces makes that index
//   unique.
// After a grid-wide barrier every CTA merges a slice of all output rows over
// the pieces of their segment: the log-sum-exp merge of the method ("LongSpec:
// Long-Context Lossless Speculative Decoding with Efficient Drafting and
// Verification", Korean summary section 2.C "aggregation"). The records of a
// slice are contiguous per piece, so one bulk copy per piece stages them in
// shared memory before the reduction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hta.h"
#include "tc_ptx.cuh"

namespace hta {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSchedB = HTA_BMAX;

struct AttnParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    const int32_t *cache_lens;
    const __nv_bfloat16 *k_spec;
    const __nv_bfloat16 *v_spec;
    const uint32_t *mask;
    void *out_o;     // bf16 or fp32 [B][T][Hq][d]
    float *out_lse;  // fp32 [B][T][Hq]
    int32_t out_fp32;
    int32_t B, T, Hq, Hkv, G, d, W;
    int64_t Lmax;
    float scale_log2;  // softmax scale * log2(e)
    int32_t R;         // packed rows per KV head = T * G
    int32_t n_rg;      // row groups per KV head
    int32_t rows_pg;   // rows per group (last group may be shorter)
    int32_t include_cache, include_tree;
    int32_t tile;          // keys per unit
    int32_t n_tree_tiles;  // ceil(T / tile) when include_tree
    // workspace
    float *ws_rec;      // [slots][rows_pg][d + 4] partial records
    unsigned int *bar;  // [0] arrivals, [1] departures
    int64_t slots;
    int32_t *dev_err;
};

// ---------------------------------------------------------------- errors

__device__ __forceinline__ void flag_error(int32_t *dev_err, int32_t f) {
    if (dev_err) atomicOr(dev_err, f);
}

// SM cycle counter: cheap to read, used to bound every wait (a read of the
// global timer costs far more and would sit on the hot wait paths)
__device__ __forceinline__ uint64_t cycles_now() { return (uint64_t)clock64(); }
constexpr uint64_t kWaitLimitCycles = 4000000000ull;  // ~2 s at 2 GHz

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- schedule

// Units of one segment of sequence b.
__device__ __forceinline__ int32_t seg_units(const AttnParams &p, int32_t Lb) {
    int32_t u = p.include_tree ? p.n_tree_tiles : 0;
    if (p.include_cache) u += (Lb + p.tile - 1) / p.tile;
    return u;
}

__device__ __forceinline__ int32_t clamp_len(const AttnParams &p, int32_t L) {
    if (L < 0 || (int64_t)L > p.Lmax) {
        flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
        L = L < 0 ? 0 : (int32_t)p.Lmax;
    }
    return L;
}

// Builds, in shared memory, the clamped lengths lens_s[b], the exclusive
// prefix pre_s[b] = sum_{b' < b} Hkv * n_rg * seg_units(b') with pre_s[B] = U,
// and the CTA boundaries lo_s[c] = floor(c * U / grid) for c = 0..grid.
// Warp 0 scans 32 sequences at a time with shuffles; every thread of the
// block must call it (it ends with __syncthreads). Bad lengths are reported
// once, by CTA 0.
__device__ inline void build_schedule(const AttnParams &p, int32_t *lens_s, int64_t *pre_s, int64_t *lo_s) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int64_t run = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int64_t v = 0;
            if (b < p.B) {
                int32_t L = p.cache_lens[b];
                if (L < 0 || (int64_t)L > p.Lmax) {
                    if (blockIdx.x == 0) flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
                    L = L < 0 ? 0 : (int32_t)p.Lmax;
                }
                lens_s[b] = L;
                v = (int64_t)p.Hkv * p.n_rg * seg_units(p, L);
            }
            int64_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (b < p.B) pre_s[b] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) pre_s[p.B] = run;
    }
    __syncthreads();
    const int64_t U = pre_s[p.B];
    for (int c = threadIdx.x; c <= (int)gridDim.x; c += blockDim.x) lo_s[c] = ((int64_t)c * U) / gridDim.x;
    __syncthreads();
}

// shared-memory bytes of the schedule arrays for B sequences and `grid` CTAs
__host__ __device__ constexpr size_t sched_bytes(int B, int grid) {
    return ((size_t)(B * 4 + 15) / 16) * 16 + (size_t)(B + 1) * 8 + (size_t)(grid + 1) * 8;
}

// CTA that owns unit u: the largest c < grid with lo_s[c] <= u (CTAs with an
// empty range share their lo with the next CTA and are never returned).
__device__ __forceinline__ int32_t cta_of_unit(int64_t u, const int64_t *lo_s, int32_t grid) {
    int32_t lo = 0, hi = grid - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (lo_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Sequence containing unit u: largest b with pre_s[b] <= u (binary search).
__device__ __forceinline__ int32_t seq_of_unit(int64_t u, const int64_t *pre_s, int32_t B) {
    int32_t lo = 0, hi = B - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (pre_s[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct UnitPos {
    int32_t b, kvh, rg;
    int64_t seg;         // segment index
    int32_t unit;        // unit index inside the segment
    int32_t seg_units;   // units in the segment
    int64_t seg_begin;   // first global unit of the segment
};

__device__ __forceinline__ UnitPos locate_unit(const AttnParams &p, int64_t u, const int32_t *lens_s,
                                               const int64_t *pre_s) {
    UnitPos r;
    r.b = seq_of_unit(u, pre_s, p.B);
    // skip sequences with zero units (several b may share pre_s)
    r.seg_units = seg_units(p, lens_s[r.b]);
    const int64_t off = u - pre_s[r.b];
    const int64_t sl = off / r.seg_units;
    r.unit = (int32_t)(off - sl * r.seg_units);
    r.kvh = (int32_t)(sl / p.n_rg);
    r.rg = (int32_t)(sl - (int64_t)r.kvh * p.n_rg);
    r.seg = ((int64_t)r.b * p.Hkv + r.kvh) * p.n_rg + r.rg;
    r.seg_begin = pre_s[r.b] + sl * r.seg_units;
    return r;
}

__device__ __forceinline__ int32_t rows_in_group(const AttnParams &p, int32_t rg) {
    int32_t r0 = rg * p.rows_pg;
    int32_t n = p.R - r0;
    return n < p.rows_pg ? n : p.rows_pg;
}

// ---------------------------------------------------------------- barrier

// Grid-wide barrier for a cooperative launch (every CTA is resident). The
// wait is bounded by ~2 s of device time; on expiry the error flag is set and
// the barrier reports failure instead of hanging. Every call returns the two
// counters to zero once the last CTA has left.
__device__ inline bool grid_barrier(const AttnParams &p) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&p.bar[0], 1u);
        const uint64_t t0 = cycles_now();
        int ok = 1;
        unsigned int v;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.bar) : "memory");
            if (v >= gridDim.x) break;
            if (cycles_now() - t0 > 2 * kWaitLimitCycles) {
                ok = 0;
                flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// Called once per CTA after its last read of data published before the
// barrier; the last CTA out resets both counters for the next call.
__device__ inline void grid_barrier_depart(const AttnParams &p) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int old = atomicAdd(&p.bar[1], 1u);
        if (old == gridDim.x - 1) {
            atomicExch(&p.bar[0], 0u);
            atomicExch(&p.bar[1], 0u);
        }
    }
}

// ---------------------------------------------------------------- partials

__device__ __forceinline__ int64_t slot_of(int64_t seg, int64_t cta) { return seg + cta; }

// ---------------------------------------------------------------- merge phase

// Merges every output row handled by this CTA. Rows are the packed rows of
// all segments, linearised segment-major and split evenly over the grid
// (the host keeps every row and unit count below 2^31, so 32-bit index math
// is exact). The CTA walks its slice in chunks of consecutive rows of one
// segment: the lanes of warp 0 bulk-copy the records of those rows from every
// piece of the segment into `buf` (one copy per piece, all in flight
// together), then one warp per row reduces them:
//   M = max_k m_k, w_k = 2^(m_k - M), O = sum_k w_k O_k / sum_k w_k l_k,
//   LSE = (M + log2 sum_k w_k l_k) ln 2.
template <int D>
__device__ inline void merge_phase(const AttnParams &p, const int32_t *lens_s, const int64_t *pre_s,
                                   const int64_t *lo_s, bool barrier_ok, uint8_t *buf, uint32_t buf_bytes) {
    constexpr int CPL = D / 32;  // columns per lane
    constexpr int REC = D + 4;   // floats per record
    constexpr uint32_t REC_BYTES = REC * 4;
    __shared__ __align__(8) uint64_t mbar;
    __shared__ int32_t ok_s;
    const uint32_t grid = gridDim.x;
    const uint32_t rows_pg = (uint32_t)p.rows_pg, n_rg = (uint32_t)p.n_rg, hkv = (uint32_t)p.Hkv;
    const uint32_t rows_total = (uint32_t)p.B * hkv * n_rg * rows_pg;
    const uint32_t r0 = (uint32_t)(((uint64_t)blockIdx.x * rows_total) / grid);
    const uint32_t r1 = (uint32_t)(((uint64_t)(blockIdx.x + 1) * rows_total) / grid);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const uint32_t bar = tc::smem_u32(&mbar);
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    uint32_t phase = 0;

    uint32_t rr = r0;
    while (rr < r1) {
        const uint32_t seg = rr / rows_pg;
        const uint32_t lr_a = rr - seg * rows_pg;
        const uint32_t sl = seg % (hkv * n_rg);  // (kvh, rg) slot inside the sequence
        const uint32_t b = seg / (hkv * n_rg);
        const uint32_t kvh = sl / n_rg, rg = sl - kvh * n_rg;
        const uint32_t nrows = (uint32_t)rows_in_group(p, (int32_t)rg);
        const uint32_t seg_stop = min(seg * rows_pg + rows_pg, r1);
        if (lr_a >= nrows) {  // padding rows of a short group
            rr = seg_stop;
            continue;
        }
        const uint32_t lr_end = min(seg_stop - seg * rows_pg, nrows);

        const int32_t su = seg_units(p, lens_s[b]);
        const int64_t sb = pre_s[b] + (int64_t)sl * su;
        int32_t c_first = 0, n_pieces = 0;
        if (su > 0 && barrier_ok) {
            c_first = cta_of_unit(sb, lo_s, (int32_t)grid);
            n_pieces = cta_of_unit(sb + su - 1, lo_s, (int32_t)grid) - c_first + 1;
        }
        const uint32_t per_row = (uint32_t)(n_pieces > 0 ? n_pieces : 1) * REC_BYTES;
        uint32_t nr = min(buf_bytes / per_row, lr_end - lr_a);
        if (nr < 1) nr = 1;  // a single row always fits: pieces <= grid

        // stage the records of rows [lr_a, lr_a + nr) of every piece
        if (warp == 0 && n_pieces > 0) {
            uint32_t mine = 0;
            for (int k = lane; k < n_pieces; k += 32) mine += lo_s[c_first + k] != lo_s[c_first + k + 1];
#pragma unroll
            for (int o = 16; o; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
            tc::fence_proxy_async_all();  // partials were written through the generic proxy
            if (lane == 0) tc::mbar_arrive_expect_tx(bar, mine * nr * REC_BYTES);
            for (int k = lane; k < n_pieces; k += 32) {
                const int32_t c = c_first + k;
                if (lo_s[c] == lo_s[c + 1]) continue;
                const float *src = p.ws_rec + ((size_t)(seg + c) * rows_pg + lr_a) * REC;
                tc::bulk_load(tc::smem_u32(buf + (uint32_t)k * nr * REC_BYTES), src, nr * REC_BYTES, bar);
            }
        }
        if (threadIdx.x == 0) {
            int ok = 1;
            if (n_pieces > 0) {
                const uint64_t t0 = cycles_now();
                while (!tc::mbar_try_wait(bar, phase)) {
                    if (cycles_now() - t0 > kWaitLimitCycles) {
                        ok = 0;
                        flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                        break;
                    }
                }
            }
            ok_s = ok;
        }
        __syncthreads();
        if (n_pieces > 0) phase ^= 1;
        const bool staged = ok_s != 0;

        for (uint32_t i = warp; i < nr; i += nwarps) {
            const uint32_t r = rg * rows_pg + lr_a + i;  // packed row
            const uint32_t t = r / (uint32_t)p.G, hq = kvh * p.G + (r - t * p.G);
            const int64_t out_row = ((int64_t)b * p.T + t) * p.Hq + hq;
            const uint8_t *row0 = buf + i * REC_BYTES;
            const uint32_t pstride = nr * REC_BYTES;  // bytes between pieces
            float M = -INFINITY, den = 0.f, acc[CPL];
#pragma unroll
            for (int k = 0; k < CPL; ++k) acc[k] = 0.f;
            for (int k0 = 0; k0 < n_pieces; k0 += 32) {
                // lane k: running max and denominator of piece k0 + k
                const int k = k0 + lane;
                float m = -INFINITY, l = 0.f;
                if (k < n_pieces && lo_s[c_first + k] != lo_s[c_first + k + 1]) {
                    const float2 ml = *reinterpret_cast<const float2 *>(row0 + (uint32_t)k * pstride + D * 4);
                    m = ml.x;
                    l = ml.y;
                }
                float Mk = m;
#pragma unroll
                for (int o = 16; o; o >>= 1) Mk = fmaxf(Mk, __shfl_xor_sync(0xffffffffu, Mk, o));
                const float Mn = fmaxf(M, Mk);
                if (Mn == -INFINITY) continue;
                // rescale what earlier groups of 32 pieces accumulated
                const float a = exp2f(M - Mn);
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc[c] *= a;
                den *= a;
                M = Mn;
                const float w = m > -INFINITY ? exp2f(m - M) : 0.f;
                float dl = w * l;
#pragma unroll
                for (int o = 16; o; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
                den += dl;
                const int nk = min(32, n_pieces - k0);
#pragma unroll 4
                for (int kk = 0; kk < nk; ++kk) {
                    const float wk = __shfl_sync(0xffffffffu, w, kk);
                    if (wk != 0.f) {
                        const float *o = reinterpret_cast<const float *>(row0 + (uint32_t)(k0 + kk) * pstride) + lane * CPL;
                        if constexpr (CPL == 4) {
                            const float4 v = *reinterpret_cast<const float4 *>(o);
                            acc[0] = fmaf(wk, v.x, acc[0]);
                            acc[1] = fmaf(wk, v.y, acc[1]);
                            acc[2] = fmaf(wk, v.z, acc[2]);
                            acc[3] = fmaf(wk, v.w, acc[3]);
                        } else {
                            const float2 v = *reinterpret_cast<const float2 *>(o);
                            acc[0] = fmaf(wk, v.x, acc[0]);
                            acc[1] = fmaf(wk, v.y, acc[1]);
                        }
                    }
                }
            }
            float lse, inv;
            if (!barrier_ok || !staged) {
                lse = __int_as_float(0x7fc00000);
                inv = __int_as_float(0x7fc00000);
            } else if (den > 0.f) {
                lse = (M + log2f(den)) * kLn2;
                inv = 1.f / den;
            } else {
                lse = -INFINITY;  // no visible key: empty softmax
                inv = 0.f;
            }
            if (p.out_fp32) {
                float *o = (float *)p.out_o + out_row * D + lane * CPL;
#pragma unroll
                for (int k = 0; k < CPL; ++k) o[k] = acc[k] * inv;
            } else {
                __nv_bfloat16 *o = (__nv_bfloat16 *)p.out_o + out_row * D + lane * CPL;
#pragma unroll
                for (int k = 0; k < CPL; k += 2)
                    *reinterpret_cast<__nv_bfloat162 *>(o + k) =
                        __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
            }
            if (lane == 0) p.out_lse[out_row] = lse;
        }
        __syncthreads();  // the buffer is reused by the next chunk
        rr = seg * rows_pg + lr_a + nr;
    }
}

}  // namespace hta
