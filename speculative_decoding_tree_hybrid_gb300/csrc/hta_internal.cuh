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
// Verification", Korean summary section 2.C "aggregation"); each thread
// loads the records of its row and column chunk straight from L2.
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
    // schedule: the unit space is split over `workers` (one CTA, or one
    // cluster of CTAs that share every tile)
    int32_t workers;
    int32_t csize;  // CTAs per cluster of the clustered tensor-core kernel (2 .. 4)
    // partial records per (segment, worker) piece: a kernel may split a piece
    // over several softmax accumulators, each written as its own record
    int32_t subs;
    // K/V storage: kv_nhd = the Hkv heads of a token are adjacent
    // ([..][rows][Hkv][d], cache and tree), else rows of a head are
    // ([..][Hkv][rows][d]); page_size 0 = one block of Lmax rows per
    // sequence, else pool pages of page_size rows named by block_table
    // [B][max_pages]. kv_generic: anything but contiguous head-major.
    int32_t kv_nhd, page_size, max_pages, num_pages, kv_generic;
    const int32_t *block_table;
    // bound of the grid-barrier wait before the merge, in SM cycles
    uint64_t bar_wait_cycles;
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

// ---------------------------------------------------------------- K/V rows

// Element offset of cache token j of sequence b, KV head kvh. A block-table
// entry outside the pool is flagged and read as page 0.
__device__ __forceinline__ int64_t cache_row_off(const AttnParams &p, int32_t b, int32_t kvh, int32_t j) {
    if (p.page_size == 0)
        return p.kv_nhd ? (((int64_t)b * p.Lmax + j) * p.Hkv + kvh) * p.d
                        : (((int64_t)b * p.Hkv + kvh) * p.Lmax + j) * p.d;
    int32_t pg = __ldg(p.block_table + (int64_t)b * p.max_pages + j / p.page_size);
    if (pg < 0 || pg >= p.num_pages) {
        flag_error(p.dev_err, HTA_DEVERR_PAGE);
        pg = 0;
    }
    const int32_t r = j % p.page_size;
    return p.kv_nhd ? (((int64_t)pg * p.page_size + r) * p.Hkv + kvh) * p.d
                    : (((int64_t)pg * p.Hkv + kvh) * p.page_size + r) * p.d;
}

// Element offset of tree token j of sequence b, KV head kvh.
__device__ __forceinline__ int64_t spec_row_off(const AttnParams &p, int32_t b, int32_t kvh, int32_t j) {
    return p.kv_nhd ? (((int64_t)b * p.T + j) * p.Hkv + kvh) * p.d
                    : (((int64_t)b * p.Hkv + kvh) * p.T + j) * p.d;
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
// and the worker boundaries lo_s[c] = floor(c * U / active) for c = 0..workers
// (c capped at `active`, the workers that get units; see below).
// Warp 0 scans 32 sequences at a time with shuffles; every thread of the
// block must call it (it ends with __syncthreads). Bad lengths are reported
// once, by CTA 0.
__device__ inline void build_schedule(const AttnParams &p, int32_t *lens_s, int64_t *pre_s, int64_t *lo_s) {
    __shared__ int32_t uniform_s;  // every sequence has the same number of units
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int64_t run = 0, v0 = 0;
        bool uniform = true;
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
            if (b0 == 0) v0 = __shfl_sync(0xffffffffu, v, 0);
            uniform = uniform && !__any_sync(0xffffffffu, b < p.B && v != v0);
            int64_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (b < p.B) pre_s[b] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            pre_s[p.B] = run;
            uniform_s = uniform ? 1 : 0;
        }
    }
    __syncthreads();
    const int64_t U = pre_s[p.B];
    // When every segment has the same number of units and the workers are
    // many more than the segments, use only a multiple of the segment count
    // (at most 1/16 of the workers left idle): each worker then covers part
    // of exactly one segment, with no switch of KV head or row group (and no
    // second record) inside its range.
    int32_t active = p.workers;
    const int64_t n_seg = (int64_t)p.B * p.Hkv * p.n_rg;
    if (uniform_s && n_seg > 0 && U > 0 && n_seg <= p.workers) {
        const int32_t aligned = (int32_t)((p.workers / n_seg) * n_seg);
        if ((p.workers - aligned) * 16 <= p.workers) active = aligned;
    }
    for (int c = threadIdx.x; c <= p.workers; c += blockDim.x)
        lo_s[c] = ((int64_t)(c < active ? c : active) * U) / active;
    __syncthreads();
}

// shared-memory bytes of the schedule arrays for B sequences and `workers` workers
__host__ __device__ constexpr size_t sched_bytes(int B, int workers) {
    return ((size_t)(B * 4 + 15) / 16) * 16 + (size_t)(B + 1) * 8 + (size_t)(workers + 1) * 8;
}

// Worker that owns unit u: the largest c < workers with lo_s[c] <= u
// (workers with an empty range share their lo with the next one and are
// never returned).
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
    // unit counts stay below 2^31 (checked on the host): 32-bit division
    const uint32_t off = (uint32_t)(u - pre_s[r.b]);
    const uint32_t sl = off / (uint32_t)r.seg_units;
    r.unit = (int32_t)(off - sl * (uint32_t)r.seg_units);
    r.kvh = (int32_t)(sl / (uint32_t)p.n_rg);
    r.rg = (int32_t)(sl - (uint32_t)r.kvh * (uint32_t)p.n_rg);
    r.seg = ((int64_t)r.b * p.Hkv + r.kvh) * p.n_rg + r.rg;
    r.seg_begin = pre_s[r.b] + (int64_t)sl * r.seg_units;
    return r;
}

__device__ __forceinline__ int32_t rows_in_group(const AttnParams &p, int32_t rg) {
    int32_t r0 = rg * p.rows_pg;
    int32_t n = p.R - r0;
    return n < p.rows_pg ? n : p.rows_pg;
}

// ---------------------------------------------------------------- barrier

// Grid-wide barrier for a persistent grid (every CTA is resident), split
// in two so that a CTA can do independent work between its arrival and the
// wait. The wait is bounded (p.bar_wait_cycles, ~4 s of device time unless a
// test sets a shorter bound); on expiry the error flag is set and the barrier
// reports failure instead of hanging. Every async copy of the CTA has
// completed before it waits here, so a CTA that gives up leaves nothing in
// flight.
// grid_barrier_depart returns the two counters to zero once the last CTA has
// left.
__device__ inline void grid_barrier_arrive(const AttnParams &p) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this CTA's partials are visible before it is counted
        atomicAdd(&p.bar[0], 1u);
    }
}

__device__ inline bool grid_barrier_wait(const AttnParams &p) {
    __shared__ int ok_s;
    if (threadIdx.x == 0) {
        const uint64_t t0 = cycles_now();
        int ok = 1;
        unsigned int v;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p.bar) : "memory");
            if (v >= gridDim.x) break;
            if (cycles_now() - t0 > p.bar_wait_cycles) {
                ok = 0;
                flag_error(p.dev_err, HTA_DEVERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
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

// Record slot of sub-accumulator x of piece (segment seg, worker w): the
// monotone staircase of pieces makes seg + w unique.
__device__ __forceinline__ int64_t slot_of(const AttnParams &p, int64_t seg, int64_t w, int32_t x = 0) {
    return (seg + w) * p.subs + x;
}

// ---------------------------------------------------------------- merge

// Pieces of segment `seg` of sequence b: the workers that cover its units
// (first worker cf, np of them, ne of them with a record; a worker with an
// empty range writes none). np = 0 for a segment without units.
struct SegPieces {
    int32_t cf, np, ne;
};

__device__ __forceinline__ SegPieces seg_pieces(const AttnParams &p, uint32_t seg, const int32_t *lens_s,
                                                const int64_t *pre_s, const int64_t *lo_s) {
    SegPieces r = {0, 0, 0};
    const uint32_t segs_per_b = (uint32_t)(p.Hkv * p.n_rg);
    const uint32_t b = seg / segs_per_b, sl = seg - b * segs_per_b;
    const int32_t su = seg_units(p, lens_s[b]);
    if (su <= 0) return r;
    const int64_t u0 = pre_s[b] + (int64_t)sl * su;
    r.cf = cta_of_unit(u0, lo_s, p.workers);
    r.np = cta_of_unit(u0 + su - 1, lo_s, p.workers) - r.cf + 1;
    for (int32_t k = 0; k < r.np; ++k) r.ne += lo_s[r.cf + k] != lo_s[r.cf + k + 1];
    return r;
}

// Folds records first, first + step, ... of one row (batches of KB, every
// load of a batch issued before any arithmetic: one round trip per batch; KB
// is set by the kernel's register budget) into the running (M, den, acc) of
// this thread's columns col0 + 64 h + e.
template <int D, int KB>
__device__ __forceinline__ void fold_records(const float *row, size_t rec_stride, int32_t nrec, bool dense,
                                             const int64_t *lo_s, int32_t cf, int32_t subs, int col0,
                                             int32_t first, int32_t step, float &M, float &den,
                                             float (&acc)[D / 16]) {
    constexpr int HPL = D / 16;
    for (int32_t k0 = first; k0 < nrec; k0 += step) {
        float2 ml[KB];
        float4 v[KB][HPL / 4];
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            const int32_t k = k0 + j;
            const bool has = k < nrec && (dense || lo_s[cf + k / subs] != lo_s[cf + k / subs + 1]);
            const float *rec = row + (size_t)k * rec_stride;
            ml[j] = has ? __ldcg(reinterpret_cast<const float2 *>(rec + D)) : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int c = 0; c < HPL / 4; ++c)
                v[j][c] = has ? __ldcg(reinterpret_cast<const float4 *>(rec + col0 + c * 64))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (ml[j].x > M) {  // a larger running max: scale what has been summed so far
                const float s = M == -INFINITY ? 0.f : tc::ex2(M - ml[j].x);
                den *= s;
#pragma unroll
                for (int c = 0; c < HPL; ++c) acc[c] *= s;
                M = ml[j].x;
            }
            const float w = ml[j].x == -INFINITY ? 0.f : tc::ex2(ml[j].x - M);  // no record: no weight
            den = fmaf(w, ml[j].y, den);
#pragma unroll
            for (int c = 0; c < HPL / 4; ++c) {
                acc[4 * c] = fmaf(w, v[j][c].x, acc[4 * c]);
                acc[4 * c + 1] = fmaf(w, v[j][c].y, acc[4 * c + 1]);
                acc[4 * c + 2] = fmaf(w, v[j][c].z, acc[4 * c + 2]);
                acc[4 * c + 3] = fmaf(w, v[j][c].w, acc[4 * c + 3]);
            }
        }
    }
}

// Normalises this thread's columns of one output row and writes them (and, in
// column chunk 0, the row's LSE); ok = false writes NaN.
template <int D>
__device__ __forceinline__ void write_item(const AttnParams &p, bool ok, float M, float den, float (&acc)[D / 16],
                                           int64_t out_row, int col0, int ch) {
    constexpr int HPL = D / 16;
    float lse, inv;
    if (!ok) {
        lse = __int_as_float(0x7fc00000);
        inv = __int_as_float(0x7fc00000);
    } else if (den > 0.f) {
        float l2;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(den));
        lse = (M + l2) * kLn2;
        inv = __frcp_rn(den);
    } else {
        lse = -INFINITY;  // no visible key: empty softmax
        inv = 0.f;
    }
    if (p.out_fp32) {
        float *op = (float *)p.out_o + out_row * D + col0;
#pragma unroll
        for (int c = 0; c < HPL; c += 4)
            *reinterpret_cast<float4 *>(op + c * 16) =
                make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
    } else {
        __nv_bfloat16 *op = (__nv_bfloat16 *)p.out_o + out_row * D + col0;
#pragma unroll
        for (int c = 0; c < HPL; c += 4) {
            const __nv_bfloat162 x = __floats2bfloat162_rn(acc[c] * inv, acc[c + 1] * inv);
            const __nv_bfloat162 y = __floats2bfloat162_rn(acc[c + 2] * inv, acc[c + 3] * inv);
            uint2 u;
            u.x = *reinterpret_cast<const uint32_t *>(&x);
            u.y = *reinterpret_cast<const uint32_t *>(&y);
            *reinterpret_cast<uint2 *>(op + c * 16) = u;
        }
    }
    if (ch == 0) p.out_lse[out_row] = lse;
}

// Merges rows [lo, lo + nrows) of segment seg over its pieces and writes O
// and LSE: one thread per (row, column chunk) reads the records of every
// piece straight from global memory (one round trip of independent loads;
// the records are L2-resident) and applies, pieces in index order, the
// log-sum-exp merge of the method ("LongSpec: Long-Context Lossless
// Speculative Decoding with Efficient Drafting and Verification", Korean
// summary section 2.C "aggregation") in its running form:
//   M = running max of m_k; when it grows, the sums so far are scaled by
//   2^(M_old - M_new); w_k = 2^(m_k - M), den += w_k l_k, acc += w_k O_k;
//   O = acc / den, LSE = (M + log2 den) ln 2.
// The result depends on the piece order only, not on which CTA merges.
// ok = false writes NaN (a piece is missing). In kernels whose batches are
// small (KB < 8), rows split over many workers are merged by up to 16
// threads per (row, column chunk), each over every S-th batch.
template <int D, int KB>
__device__ inline void merge_rows(const AttnParams &p, const int64_t *lo_s, uint32_t seg, const SegPieces &pc,
                                  uint32_t lo, uint32_t nrows_run, bool ok) {
    constexpr int HPL = D / 16;  // output columns per thread
    constexpr int REC = D + 4;   // floats per record: O | m | l | w | pad
    constexpr int NCH = D / HPL; // column chunks per row (16)
    const uint32_t rows_pg = (uint32_t)p.rows_pg, n_rg = (uint32_t)p.n_rg;
    const uint32_t segs_per_b = (uint32_t)p.Hkv * n_rg;
    const uint32_t G = (uint32_t)p.G, T = (uint32_t)p.T, Hq = (uint32_t)p.Hq;
    const int32_t subs = p.subs, cf = pc.cf, nrec = pc.np * subs;
    const bool dense = pc.ne == pc.np;  // every piece has a record: no per-piece checks below
    const uint32_t b = seg / segs_per_b, sl = seg - b * segs_per_b;
    const uint32_t kvh = sl / n_rg, rg = sl - kvh * n_rg;
    // record x of piece k, row lr: ws_rec + ((seg + cf + k) * subs + x) * rows_pg + lr) * REC
    const float *const rec0 = p.ws_rec + ((size_t)(seg + cf) * subs * rows_pg) * REC;
    const size_t rec_stride = (size_t)rows_pg * REC;  // floats between consecutive records
    const int32_t items = (int32_t)nrows_run * NCH;
    if constexpr (KB >= 8) {
        // one thread per item: a batch holds every piece of the shapes these kernels take
        for (int32_t item = threadIdx.x; item < items; item += blockDim.x) {
            const int32_t i = item / NCH, ch = item - i * NCH;
            const uint32_t lr = lo + (uint32_t)i;
            const uint32_t r = rg * rows_pg + lr;  // packed row within the KV head
            const uint32_t t = r / G, hq = kvh * G + (r - t * G);
            const int64_t out_row = ((int64_t)b * T + t) * Hq + hq;
            const int col0 = ch * 4;  // this thread's columns: col0 + 64 h + e, h < HPL / 4, e < 4
            float M = -INFINITY, den = 0.f, acc[HPL];
#pragma unroll
            for (int c = 0; c < HPL; ++c) acc[c] = 0.f;
            if (ok) fold_records<D, KB>(rec0 + (size_t)lr * REC, rec_stride, nrec, dense, lo_s, cf, subs, col0, 0, KB, M,
                                        den, acc);
            write_item<D>(p, ok, M, den, acc, out_row, col0, ch);
        }
    } else {
        // Few items and many records (rows split over many workers): S threads
        // per item, neighbouring lanes, each folding every S-th batch of
        // records; their partial states are combined by shuffles in a fixed
        // order, so the result is still deterministic.
        int32_t S = 1;
        while (S < 16 && items * S * 2 <= (int32_t)blockDim.x && S * KB < nrec) S *= 2;
        const int32_t span = (items * S + 31) & ~31;  // whole warps: every lane takes part in the shuffles
        for (int32_t slot = threadIdx.x; slot < span; slot += blockDim.x) {
            const int32_t item = slot / S, sub = slot - item * S;
            const bool live = item < items;
            const int32_t i = live ? item / NCH : 0, ch = live ? item - i * NCH : 0;
            const uint32_t lr = lo + (uint32_t)i;
            const uint32_t r = rg * rows_pg + lr;
            const uint32_t t = r / G, hq = kvh * G + (r - t * G);
            const int64_t out_row = ((int64_t)b * T + t) * Hq + hq;
            const int col0 = ch * 4;
            float M = -INFINITY, den = 0.f, acc[HPL];
#pragma unroll
            for (int c = 0; c < HPL; ++c) acc[c] = 0.f;
            if (ok && live)
                fold_records<D, KB>(rec0 + (size_t)lr * REC, rec_stride, nrec, dense, lo_s, cf, subs, col0, sub * KB,
                                    S * KB, M, den, acc);
            for (int o = S >> 1; o > 0; o >>= 1) {  // S is the same in every thread
                const float M2 = __shfl_xor_sync(0xffffffffu, M, o);
                const float d2 = __shfl_xor_sync(0xffffffffu, den, o);
                const float Mn = fmaxf(M, M2);
                const float s1 = M == -INFINITY ? 0.f : tc::ex2(M - Mn);
                const float s2 = M2 == -INFINITY ? 0.f : tc::ex2(M2 - Mn);
                den = fmaf(den, s1, d2 * s2);
#pragma unroll
                for (int c = 0; c < HPL; ++c) {
                    const float a2 = __shfl_xor_sync(0xffffffffu, acc[c], o);
                    acc[c] = fmaf(acc[c], s1, a2 * s2);
                }
                M = Mn;
            }
            if (live && sub == 0) write_item<D>(p, ok, M, den, acc, out_row, col0, ch);
        }
    }
}

// Merges every output row handled by this CTA, after a grid-wide barrier
// that it enters here (persistent grids, every CTA resident). Rows are the
// packed rows of all segments, linearised segment-major and split evenly
// over the grid (the host keeps every row and unit count below 2^31, so
// 32-bit index math is exact). The CTA's slice is cut into runs, one per
// segment it touches; between its arrival at the barrier and the wait, one
// thread per run locates the run's pieces, so that index math overlaps the
// barrier; each run is then merged by merge_rows.
// `buf` is idle shared memory for the run table; the block has more than
// kMergeRuns threads. `arrived`: this CTA has already arrived on the barrier.
constexpr int kMergeRuns = 64;

template <int D, int KB>
__device__ inline void merge_phase(const AttnParams &p, const int32_t *lens_s, const int64_t *pre_s,
                                   const int64_t *lo_s, uint8_t *buf, bool arrived = false) {
    const uint32_t grid = gridDim.x;
    const uint32_t rows_pg = (uint32_t)p.rows_pg, n_rg = (uint32_t)p.n_rg, hkv = (uint32_t)p.Hkv;
    const uint32_t segs_per_b = hkv * n_rg;
    const uint32_t rows_total = (uint32_t)p.B * segs_per_b * rows_pg;
    const uint32_t r0 = (uint32_t)(((uint64_t)blockIdx.x * rows_total) / grid);
    const uint32_t r1 = (uint32_t)(((uint64_t)(blockIdx.x + 1) * rows_total) / grid);
    int32_t *run_seg = reinterpret_cast<int32_t *>(buf);
    int32_t *run_cf = run_seg + kMergeRuns;  // first piece (worker index)
    int32_t *run_np = run_cf + kMergeRuns;   // pieces
    int32_t *run_lo = run_np + kMergeRuns;   // first local row
    int32_t *run_nr = run_lo + kMergeRuns;   // rows
    int32_t *run_ne = run_nr + kMergeRuns;   // pieces with a record
    if (!arrived) grid_barrier_arrive(p);
    else __syncthreads();
    bool ok = true, waited = false;
    const uint32_t seg_lo = r0 / rows_pg, seg_end = r1 > r0 ? (r1 - 1) / rows_pg + 1 : seg_lo;
    for (uint32_t sb = seg_lo; sb < seg_end || !waited; sb += kMergeRuns) {
        const uint32_t n_runs = sb < seg_end ? min((uint32_t)kMergeRuns, seg_end - sb) : 0u;
        if (threadIdx.x < n_runs) {
            const uint32_t seg = sb + threadIdx.x;
            const uint32_t sl = seg % segs_per_b;
            const uint32_t nrows = (uint32_t)rows_in_group(p, (int32_t)(sl % n_rg));
            const uint32_t base = seg * rows_pg;
            const uint32_t lo = (r0 > base ? r0 : base) - base;
            const uint32_t hi = min(r1 - base, nrows);
            SegPieces pc = {0, 0, 0};
            if (hi > lo) pc = seg_pieces(p, seg, lens_s, pre_s, lo_s);
            run_seg[threadIdx.x] = (int32_t)seg;
            run_cf[threadIdx.x] = pc.cf;
            run_np[threadIdx.x] = pc.np;
            run_lo[threadIdx.x] = (int32_t)lo;
            run_nr[threadIdx.x] = hi > lo ? (int32_t)(hi - lo) : 0;
            run_ne[threadIdx.x] = pc.ne;
        }
        if (!waited) {
            ok = grid_barrier_wait(p);  // its closing __syncthreads also publishes the table
            waited = true;
        } else {
            __syncthreads();
        }
        for (uint32_t j = 0; j < n_runs; ++j) {
            const SegPieces pc = {run_cf[j], run_np[j], run_ne[j]};
            merge_rows<D, KB>(p, lo_s, (uint32_t)run_seg[j], pc, (uint32_t)run_lo[j], (uint32_t)run_nr[j], ok);
        }
        __syncthreads();  // the run table is rewritten by the next batch
    }
}

}  // namespace hta
