// LogitSpec draft-tree builder ("LogitSpec: Accelerating Retrieval-based
// Speculative Decoding via Next Next Token Speculation", section 2, workflow
// steps 1 and 2): from the target's last logits and the sequence's token
// history, build the draft tree that the verification step checks.
//
//   x_{i+1}   = the largest logit (ties: the smaller token id)
//   guesses   = the next k logits in that order (next-next token guesses)
//   g1        = (x_{i-m+2}, ..., x_i, x_{i+1})           one query
//   g2(r)     = (x_{i-m+3}, ..., x_i, x_{i+1}, guess_r)  one query per guess
// Each query is looked up in the history: its latest occurrence at s with a
// token after it (s + m <= len - 1). The tree: node 0 = x_{i+1}; then up to
// keep[0] tokens after g1's match as a chain under the root; then for each
// guess r in rank order, the guess as a child of the root and up to keep[r]
// tokens after g2(r)'s match as a chain under it; nodes are added until T,
// unused nodes are padding (parent 0, token -1).
//
// One cluster of 4 CTAs (512 threads each) per sequence; the leader CTA
// holds the selection and the tree, the others add bandwidth:
//  1. top-(k+1) of the logits by radix select on an order-preserving integer
//     key: an 11-bit histogram of every key (each CTA a quarter of the
//     logits, summed by the leader over distributed shared memory), then one
//     pass keeping the keys above the chosen digit and moving the keys at it
//     into the leader's shared memory (four 16-byte loads in flight per
//     thread). When those are few (at most kDirect: a few hundred for
//     N(0, 1)-like logits) one counting rank over them all, key descending
//     and id ascending, gives the k+1 survivors in order; otherwise three
//     more digits resolve the threshold, the keys above it and the smallest
//     tied ids are the survivors, ranked by a counting sort (near-equal
//     logits too many for shared memory resolve with passes over the logits);
//  2. the 1 + k queries go into a hash table in shared memory (the pages'
//     hash-based lookup, copied to every CTA of the cluster) and every
//     history position (a quarter per CTA) hashes its m-gram once, tests a
//     bitmap of the query hashes (most positions stop there), probes the
//     table, confirms a hit token by token and keeps the latest start per
//     query (atomicMax in the leader);
//  3. branch r starts at min(1 + the sizes the branches before it want, T):
//     one warp scans the (at most 65) branch sizes, then every thread writes
//     its nodes, finding its branch by binary search.
#include <cooperative_groups.h>

#include "hta_internal.cuh"
#include "hta_launch.h"

namespace cg = cooperative_groups;

namespace hta {
namespace {

constexpr int kThreads = 512;
constexpr int kCtas = 4;  // CTAs per sequence: a thread-block cluster
constexpr int kWarps = kThreads / 32;
constexpr int kTable = 256;  // hash slots (at least twice the queries)
constexpr int kBloom = 4096; // bits of the query-hash bitmap that screens history positions
constexpr int kEqCap = 512;  // threshold ties gathered in one pass (more: the ordered scan)
constexpr int kBuf = 1024;   // keys of the first digit held in shared memory
constexpr int kDirect = kThreads / 2;  // candidates ranked directly (two threads per key)

// order-preserving key: a larger float gives a larger key; -0 counts as +0
// and NaN ranks below every number
__device__ __forceinline__ uint32_t fkey(float x) {
    uint32_t u = __float_as_uint(x);
    if (x != x) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Calls f(i, key) for every logit, four 16-byte loads in flight per thread
// when the row is 16-byte aligned (else four scalar loads).
template <class F>
__device__ __forceinline__ void for_each_key(const float *lg, int V, F f) {
    if ((V & 3) == 0 && ((uintptr_t)lg & 15u) == 0) {
        const float4 *v4 = reinterpret_cast<const float4 *>(lg);
        const int n4 = V >> 2;
        for (int i = threadIdx.x; i < n4; i += 4 * kThreads) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = i + u * kThreads;
                if (j < n4) x[u] = __ldg(v4 + j);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = i + u * kThreads;
                if (j < n4) {
                    f(4 * j, fkey(x[u].x));
                    f(4 * j + 1, fkey(x[u].y));
                    f(4 * j + 2, fkey(x[u].z));
                    f(4 * j + 3, fkey(x[u].w));
                }
            }
        }
    } else {
        for (int i = threadIdx.x; i < V; i += 4 * kThreads) {
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = i + u * kThreads;
                if (j < V) x[u] = __ldg(lg + j);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = i + u * kThreads;
                if (j < V) f(j, fkey(x[u]));
            }
        }
    }
}

// FNV-1a over the first m (<= HTA_LSPEC_MMAX) token ids; unrolled and
// predicated so that an array argument stays in registers
__device__ __forceinline__ uint32_t gram_hash(const int32_t (&t)[HTA_LSPEC_MMAX], int m) {
    uint32_t h = 2166136261u;
#pragma unroll
    for (int i = 0; i < HTA_LSPEC_MMAX; ++i)
        if (i < m) h = (h ^ (uint32_t)t[i]) * 16777619u;
    return h;
}

// All threads: the digit d of `hist` (nbins <= 4 * kThreads bins) holding the
// need-th largest key counted from the top bin, and how many keys of d are
// still needed; written to *d_out, *need_out. A suffix scan over the bins:
// thread t owns bins nbins-1-c*t .. nbins-c*(t+1) (c = bins per thread).
__device__ __forceinline__ void select_digit(const uint32_t *hist, int nbins, int32_t need, int32_t *wsum,
                                             int32_t *d_out, int32_t *need_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = (nbins + kThreads - 1) / kThreads;
    int32_t mine = 0;
    for (int j = 0; j < c; ++j) {
        const int bin = nbins - 1 - (tid * c + j);
        if (bin >= 0) mine += (int32_t)hist[bin];
    }
    int32_t incl = mine;  // inclusive scan over the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int32_t before = incl - mine;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    if (before < need && need <= before + mine) {
        int32_t left = need - before;
        for (int j = 0; j < c; ++j) {
            const int bin = nbins - 1 - (tid * c + j);
            if (bin < 0) break;
            if ((int32_t)hist[bin] >= left) {
                *d_out = bin;
                *need_out = left;
                break;
            }
            left -= (int32_t)hist[bin];
        }
    }
    __syncthreads();
}

struct LspecSmem {
    uint32_t hist[kWarps][256];
    uint32_t cand_key[HTA_LSPEC_KMAX + 1];
    int32_t cand_id[HTA_LSPEC_KMAX + 1];
    int32_t top[HTA_LSPEC_KMAX + 1];  // ranked token ids
    int32_t q[HTA_LSPEC_KMAX + 1][HTA_LSPEC_MMAX];
    int32_t q_ok[HTA_LSPEC_KMAX + 1];
    int32_t best[HTA_LSPEC_KMAX + 1];
    uint32_t slot_hash[kTable];
    uint32_t bloom[kBloom / 32];  // bit h % kBloom set for every query hash h
    int32_t slot_q[kTable];
    int32_t br_start[HTA_LSPEC_KMAX + 1], br_len[HTA_LSPEC_KMAX + 1];
    int32_t wcount[kWarps];
    int32_t eq_id[kEqCap > kBuf ? kEqCap : kBuf];
    uint32_t buf_key[kBuf];
    int32_t buf_id[kBuf];
    uint32_t prefix, mask;
    int32_t remaining, sel_d, n_cand, n_buf, n_eq, eq_total, eq_base, n_nodes;
};

__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads)
    k_logitspec_tree(const __grid_constant__ LspecParams p) {
    __shared__ LspecSmem sm;
    cg::cluster_group cl = cg::this_cluster();
    const unsigned rank = cl.block_rank();
    LspecSmem &lead = *cl.map_shared_rank(&sm, 0);  // the leader's shared memory
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / kCtas;
    const int K = p.k + 1, m = p.m;
    const float *lg = p.logits + (int64_t)b * p.V;
    const int32_t *hs = p.hist + (int64_t)b * p.Lh_max;
    int64_t n = p.hist_len[b];
    if (n < 0 || n > p.Lh_max) {
        if (rank == 0 && tid == 0) flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
        n = n < 0 ? 0 : p.Lh_max;
    }
    // this CTA's slice of the logits (a multiple of 4 long: 16-byte loads stay aligned)
    const int chunk = ((p.V + kCtas - 1) / kCtas + 3) & ~3;
    const int v_lo = min(p.V, (int)rank * chunk), v_hi = min(p.V, v_lo + chunk);

    // ---- 1. the K largest keys: radix select of the K-th largest key.
    // Pass 0 histograms the top 11 bits of every key (global); one more global
    // pass then keeps the keys above that digit (fewer than K) and moves the
    // keys at it to shared memory when they fit (a few hundred for
    // N(0, 1)-like logits), where the remaining 21 bits are resolved. Keys
    // that do not fit (many near-equal logits) resolve with global passes.
    uint32_t *h2k = &sm.hist[0][0];  // 2048 bins for pass 0
    for (int i = tid; i < 2048; i += kThreads) h2k[i] = 0u;
    if (tid == 0) {
        sm.n_cand = 0;
        sm.n_buf = 0;
        sm.n_eq = 0;
        sm.eq_base = 0;
    }
    __syncthreads();
    for_each_key(lg + v_lo, v_hi - v_lo, [&](int, uint32_t key) { atomicAdd(&h2k[key >> 21], 1u); });
    cl.sync();  // every slice's histogram is complete
    if (rank == 0) {
        for (int i = tid; i < 2048; i += kThreads) {
            uint32_t c = h2k[i];
            for (unsigned r = 1; r < kCtas; ++r) c += cl.map_shared_rank(h2k, r)[i];
            h2k[i] = c;
        }
        __syncthreads();
        select_digit(h2k, 2048, K, sm.wcount, &sm.sel_d, &sm.remaining);
        if (tid == 0) {
            sm.prefix = (uint32_t)sm.sel_d << 21;
            sm.mask = 0xFFE00000u;
            sm.eq_total = (int32_t)h2k[sm.sel_d];  // keys in the chosen digit
        }
    }
    cl.sync();  // the first digit is in the leader
    const bool in_smem = lead.eq_total <= kBuf;
    {
        const uint32_t d1 = lead.prefix >> 21;
        for_each_key(lg + v_lo, v_hi - v_lo, [&](int i, uint32_t key) {
            const uint32_t top = key >> 21;
            if (top > d1) {
                const int slot = atomicAdd(&lead.n_cand, 1);
                lead.cand_key[slot] = key;
                lead.cand_id[slot] = v_lo + i;
            } else if (top == d1 && in_smem) {
                const int slot = atomicAdd(&lead.n_buf, 1);
                lead.buf_key[slot] = key;
                lead.buf_id[slot] = v_lo + i;
            }
        });
    }
    cl.sync();  // every candidate is in the leader
    if (rank == 0) {
    const int32_t n_c0 = sm.n_cand, n_b0 = sm.n_buf;
    if (in_smem && n_c0 + n_b0 <= kDirect) {
        // every key above the first digit is a candidate and every key of the
        // digit is in the buffer: rank them all at once, key descending and
        // id ascending, two threads per key (each over half of the keys)
        const int32_t n_all = n_c0 + n_b0;
        for (int e = tid; e < n_c0; e += kThreads) {
            sm.buf_key[n_b0 + e] = sm.cand_key[e];
            sm.buf_id[n_b0 + e] = sm.cand_id[e];
        }
        __syncthreads();
        const int e = tid >> 1, h = tid & 1;
        int32_t pos = 0, id = 0;
        if (e < n_all) {
            const uint32_t ky = sm.buf_key[e];
            id = sm.buf_id[e];
#pragma unroll 4
            for (int g = h; g < n_all; g += 2) {
                const uint32_t kg = sm.buf_key[g];
                pos += (kg > ky) || (kg == ky && sm.buf_id[g] < id);
            }
        }
        pos += __shfl_xor_sync(0xffffffffu, pos, 1);
        if (e < n_all && h == 0 && pos < K) sm.top[pos] = id;
        __syncthreads();
    } else {
        // the low 21 bits in three digits (8, 8, 5), over the buffer or the logits
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = pass == 0 ? 13 : pass == 1 ? 5 : 0;
            const uint32_t dmask = pass == 2 ? 31u : 255u;
            for (int i = tid; i < kWarps * 256; i += kThreads) (&sm.hist[0][0])[i] = 0u;
            __syncthreads();
            const uint32_t prefix = sm.prefix, mask = sm.mask;
            auto count = [&](int, uint32_t key) {
                if ((key & mask) == prefix) atomicAdd(&sm.hist[warp][(key >> shift) & dmask], 1u);
            };
            if (in_smem) {
                for (int e = tid; e < sm.n_buf; e += kThreads) count(0, sm.buf_key[e]);
            } else {
                for_each_key(lg, p.V, count);
            }
            __syncthreads();
            if (tid < 256) {  // fold the warps' histograms into row 0
                uint32_t c = 0;
                for (int w = 0; w < kWarps; ++w) c += sm.hist[w][tid];
                sm.hist[0][tid] = c;
            }
            __syncthreads();
            // the digit holding the remaining-th largest key, from the top
            const int32_t need_in = sm.remaining;
            __syncthreads();
            select_digit(&sm.hist[0][0], (int)dmask + 1, need_in, sm.wcount, &sm.sel_d, &sm.remaining);
            if (tid == 0) {
                const int32_t d = sm.sel_d;
                if (pass == 2) sm.eq_total = (int32_t)sm.hist[0][d];  // every key equal to the threshold
                sm.prefix |= (uint32_t)d << shift;
                sm.mask |= dmask << shift;
            }
            __syncthreads();
        }
        const uint32_t thr = sm.prefix;
        const int32_t need_eq = sm.remaining;
        if (in_smem) {
            // the buffer's keys above the threshold, then the need_eq smallest tied ids
            for (int e = tid; e < sm.n_buf; e += kThreads) {
                const uint32_t key = sm.buf_key[e];
                if (key > thr) {
                    const int slot = atomicAdd(&sm.n_cand, 1);
                    sm.cand_key[slot] = key;
                    sm.cand_id[slot] = sm.buf_id[e];
                } else if (key == thr) {
                    sm.eq_id[atomicAdd(&sm.n_eq, 1)] = sm.buf_id[e];
                }
            }
            __syncthreads();
        } else if (sm.eq_total <= kEqCap) {
            // one more global pass: the keys above the threshold below the first
            // digit were not kept yet, and every tie at it
            const uint32_t d1 = thr >> 21;
            for_each_key(lg, p.V, [&](int i, uint32_t key) {
                if (key > thr && (key >> 21) == d1) {
                    const int slot = atomicAdd(&sm.n_cand, 1);
                    sm.cand_key[slot] = key;
                    sm.cand_id[slot] = i;
                } else if (key == thr) {
                    sm.eq_id[atomicAdd(&sm.n_eq, 1)] = i;
                }
            });
            __syncthreads();
        }
        if (in_smem || sm.eq_total <= kEqCap) {
            const int n_eq = sm.n_eq, base = sm.n_cand;
            for (int e = tid; e < n_eq; e += kThreads) {
                const int32_t id = sm.eq_id[e];
                int32_t rank = 0;
                for (int f = 0; f < n_eq; ++f) rank += sm.eq_id[f] < id;
                if (rank < need_eq) {
                    sm.cand_key[base + rank] = thr;
                    sm.cand_id[base + rank] = id;
                }
            }
            __syncthreads();
        } else {
            for (int i0 = 0; i0 < p.V; i0 += kThreads) {
                // many ties: the ordered scan takes the need_eq smallest tied ids,
                // counting ties chunk by chunk in id order (keys above the
                // threshold inside the first digit join on the way)
                const int i = i0 + tid;
                const uint32_t key = i < p.V ? fkey(lg[i]) : 0u;
                if (i < p.V && key > thr && (key >> 21) == (thr >> 21)) {
                    const int slot = atomicAdd(&sm.n_cand, 1);
                    sm.cand_key[slot] = key;
                    sm.cand_id[slot] = i;
                }
                const int32_t eq_base = sm.eq_base;  // uniform: written only between the barriers below
                if (eq_base < need_eq) {
                    const bool eq = i < p.V && key == thr;
                    const unsigned bal = __ballot_sync(0xffffffffu, eq);
                    if (lane == 0) sm.wcount[warp] = __popc(bal);
                    __syncthreads();
                    int32_t before = eq_base;
                    for (int w = 0; w < warp; ++w) before += sm.wcount[w];
                    const int32_t rank = before + __popc(bal & ((1u << lane) - 1u));
                    if (eq && rank < need_eq) {
                        const int slot = atomicAdd(&sm.n_cand, 1);
                        sm.cand_key[slot] = key;
                        sm.cand_id[slot] = i;
                    }
                    __syncthreads();
                    if (tid == 0) {
                        int32_t tot = 0;
                        for (int w = 0; w < kWarps; ++w) tot += sm.wcount[w];
                        sm.eq_base = eq_base + tot;
                    }
                    __syncthreads();
                }
            }
            __syncthreads();
        }
        // rank sort: key descending, id ascending
        if (tid < K) {
            const uint32_t ky = sm.cand_key[tid];
            const int32_t id = sm.cand_id[tid];
            int32_t pos = 0;
            for (int j = 0; j < K; ++j) {
                const uint32_t kj = sm.cand_key[j];
                pos += (kj > ky) || (kj == ky && sm.cand_id[j] < id);
            }
            sm.top[pos] = id;
        }
        __syncthreads();
    }
    const int32_t x1 = sm.top[0];

    // ---- 2. queries into the hash table (leader), one scan of the history (cluster)
    for (int i = tid; i < kTable; i += kThreads) sm.slot_q[i] = -1;
    for (int i = tid; i < kBloom / 32; i += kThreads) sm.bloom[i] = 0u;
    if (tid < K) {
        // query 0: the last m-1 history tokens and x1; query r: the last m-2, x1, guess r
        const int r = tid, hist_part = r == 0 ? m - 1 : m - 2;
        const bool ok = n >= hist_part;
        sm.q_ok[r] = ok;
        sm.best[r] = -1;
        if (ok) {
            for (int j = 0; j < hist_part; ++j) sm.q[r][j] = hs[n - hist_part + j];
            sm.q[r][hist_part] = x1;
            if (r > 0) sm.q[r][m - 1] = sm.top[r];
        }
    }
    __syncthreads();
    if (tid < K && sm.q_ok[tid]) {  // each query claims a slot (linear probing)
        const uint32_t h = gram_hash(sm.q[tid], m);
        uint32_t s = h & (kTable - 1);
        while (atomicCAS(&sm.slot_q[s], -1, tid) != -1) s = (s + 1) & (kTable - 1);
        sm.slot_hash[s] = h;
        atomicOr(&sm.bloom[(h >> 5) & (kBloom / 32 - 1)], 1u << (h & 31));
    }
    }  // leader
    cl.sync();  // the queries and their table are in the leader
    if (rank != 0) {  // a local copy of the table and the queries
        for (int i = tid; i < kTable; i += kThreads) {
            sm.slot_q[i] = lead.slot_q[i];
            sm.slot_hash[i] = lead.slot_hash[i];
        }
        for (int i = tid; i < kBloom / 32; i += kThreads) sm.bloom[i] = lead.bloom[i];
        for (int i = tid; i < K * HTA_LSPEC_MMAX; i += kThreads) (&sm.q[0][0])[i] = (&lead.q[0][0])[i];
    }
    __syncthreads();
    // this CTA's quarter of the positions; four per thread and iteration,
    // their tokens loaded together into registers (a position's m-gram: the
    // next m tokens, m <= 8)
    const int64_t n_pos = n - m > 0 ? n - m : 0;  // starts s with s + m <= n - 1
    const int64_t pchunk = (n_pos + kCtas - 1) / kCtas;
    const int64_t s_lo = min(n_pos, (int64_t)rank * pchunk), s_hi = min(n_pos, s_lo + pchunk);
    for (int64_t s0 = s_lo + tid; s0 < s_hi; s0 += 4 * kThreads) {
        int32_t g[4][HTA_LSPEC_MMAX];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t s = s0 + (int64_t)u * kThreads;
#pragma unroll
            for (int j = 0; j < HTA_LSPEC_MMAX; ++j) g[u][j] = (j < m && s < s_hi) ? __ldg(hs + s + j) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t s = s0 + (int64_t)u * kThreads;
            if (s >= s_hi) continue;
            const uint32_t h = gram_hash(g[u], m);
            // most positions match no query's hash: one bitmap test, no probe
            if (!((sm.bloom[(h >> 5) & (kBloom / 32 - 1)] >> (h & 31)) & 1u)) continue;
            for (uint32_t t = h & (kTable - 1); sm.slot_q[t] >= 0; t = (t + 1) & (kTable - 1)) {
                if (sm.slot_hash[t] != h) continue;
                const int r = sm.slot_q[t];
                bool same = true;
#pragma unroll
                for (int j = 0; j < HTA_LSPEC_MMAX; ++j) same = same && (j >= m || g[u][j] == sm.q[r][j]);
                if (same) atomicMax(&lead.best[r], (int32_t)s);
            }
        }
    }
    cl.sync();  // every match is in the leader
    if (rank != 0) return;

    // ---- 3. tree layout, then the nodes
    const int32_t x1 = sm.top[0];
    if (warp == 0) {
        // branch r starts at min(1 + the sizes wanted before it, T): a scan
        // over the branches, 32 at a time
        int32_t carry = 1;  // the root
        for (int r0 = 0; r0 < K; r0 += 32) {
            const int r = r0 + lane;
            int32_t want = 0;
            if (r < K) {
                int32_t len = 0;
                if (sm.best[r] >= 0) {
                    const int64_t avail = n - ((int64_t)sm.best[r] + m);
                    len = (int32_t)min((int64_t)p.keep[r], avail);
                }
                want = len + (r > 0 ? 1 : 0);  // a guess node heads its branch
            }
            int32_t incl = want;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            if (r < K) {
                const int32_t start = min(carry + incl - want, p.T), end = min(carry + incl, p.T);
                sm.br_start[r] = start;
                sm.br_len[r] = end - start;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) sm.n_nodes = min(carry, p.T);
    }
    __syncthreads();
    const int32_t nn = sm.n_nodes;
    int32_t *par = p.parents + (int64_t)b * p.T;
    int32_t *tok = p.tokens + (int64_t)b * p.T;
    for (int v = tid; v < p.T; v += kThreads) {
        int32_t pv = 0, tv = -1;  // padding
        if (v == 0) {
            pv = -1;
            tv = x1;
        } else if (v < nn) {
            int r = 0, hi = K - 1;  // the branch holding node v: the last one starting at or before v
            while (r < hi) {
                const int mid = (r + hi + 1) >> 1;
                if (sm.br_start[mid] <= v) r = mid;
                else hi = mid - 1;
            }
            const int32_t j = v - sm.br_start[r];
            if (r > 0 && j == 0) {
                tv = sm.top[r];  // the guess itself, a child of the root
            } else {
                const int32_t off = r > 0 ? j - 1 : j;
                tv = hs[sm.best[r] + m + off];
                pv = j == 0 ? 0 : v - 1;
            }
            if (r > 0 && j == 0) pv = 0;
        }
        par[v] = pv;
        tok[v] = tv;
    }
    if (tid == 0) {
        p.n_nodes[b] = nn;
        p.next_token[b] = x1;
    }
}

}  // namespace

cudaError_t lspec_launch(const LspecParams &p, cudaStream_t stream) {
    k_logitspec_tree<<<p.B * kCtas, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace hta
