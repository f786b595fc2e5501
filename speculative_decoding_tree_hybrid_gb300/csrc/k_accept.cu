// Accept walk and KV commit: the step after tree verification.
//
// The draft tree is rooted at the target's own next token ("LogitSpec:
// Accelerating Retrieval-based Speculative Decoding via Next Next Token
// Speculation", section 2, workflow step 2), and verification yields, for
// every node, the target's greedy prediction of the token after it. Greedy
// acceptance: the root (node 0) is accepted; a child of the last accepted node
// is accepted when its draft token equals the target's prediction at that
// node (the smallest such child index); the walk stops at the first node
// without one. The accepted nodes' K/V rows are then appended to their
// sequence's cache at L_b, L_b + 1, ... and cache_lens[b] grows by the count
// (clamped so that nothing is written past Lmax; a clamp sets
// HTA_DEVERR_CACHE_LEN).
//
// One CTA per sequence. Warp 0 walks the tree from shared memory, 32
// candidate children per ballot; then all threads copy the path's rows in
// 16-byte chunks, eight loads in flight per thread. kGeneric: the cache (and
// the tree's K/V) in another storage than contiguous head-major (token-major
// rows, pool pages named by a block table); a row whose page entry lies
// outside the pool is not written and flags HTA_DEVERR_PAGE.
#include "hta_launch.h"

namespace hta {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;

// Row index (in rows of d elements) of cache token pos of (b, h) under `st`;
// -1 when its page entry lies outside the pool.
__device__ __forceinline__ int64_t store_row(const KvStore &st, int b, int h, int64_t pos, int Hkv, int64_t Lmax) {
    if (st.page_size == 0)
        return st.nhd ? ((int64_t)b * Lmax + pos) * Hkv + h : ((int64_t)b * Hkv + h) * Lmax + pos;
    const int32_t pg = __ldg(st.block_table + (int64_t)b * st.max_pages + pos / st.page_size);
    if (pg < 0 || pg >= st.num_pages) return -1;
    const int64_t r = pos % st.page_size;
    return st.nhd ? ((int64_t)pg * st.page_size + r) * Hkv + h : ((int64_t)pg * Hkv + h) * st.page_size + r;
}

template <bool kGeneric>
__global__ void __launch_bounds__(kThreads)
    k_accept_commit(const int32_t *__restrict__ parents, const int32_t *__restrict__ draft,
                    const int32_t *__restrict__ target, int T, int Hkv, int d, int64_t Lmax,
                    const uint4 *__restrict__ k_spec, const uint4 *__restrict__ v_spec, uint4 *k_cache,
                    uint4 *v_cache, int32_t *cache_lens, int32_t *accepted, int32_t *n_accepted,
                    int32_t *next_token, int32_t *dev_err, const KvStore st) {
    __shared__ int32_t par_s[HTA_TMAX], tok_s[HTA_TMAX], tgt_s[HTA_TMAX], path_s[HTA_TMAX];
    __shared__ int32_t n_s, len_s;
    const int b = blockIdx.x, tid = threadIdx.x;
    for (int i = tid; i < T; i += kThreads) {
        par_s[i] = parents[(int64_t)b * T + i];
        tok_s[i] = draft[(int64_t)b * T + i];
        tgt_s[i] = target[(int64_t)b * T + i];
    }
    if (tid == 0) {
        int32_t L = cache_lens[b];
        if (L < 0 || (int64_t)L > Lmax) {
            flag_error(dev_err, HTA_DEVERR_CACHE_LEN);
            L = L < 0 ? 0 : (int32_t)Lmax;
        }
        len_s = L;
    }
    __syncthreads();
    if (tid < 32) {
        const int lane = tid;
        int cur = 0, n = 1;
        if (lane == 0) path_s[0] = 0;
        for (;;) {
            const int32_t want = tgt_s[cur];
            int next = -1;
            for (int base = cur + 1; base < T && next < 0; base += 32) {
                const int c = base + lane;
                const unsigned hit = __ballot_sync(0xffffffffu, c < T && par_s[c] == cur && tok_s[c] == want);
                if (hit) next = base + __ffs(hit) - 1;
            }
            if (next < 0) break;
            if (lane == 0) path_s[n] = next;
            ++n;
            cur = next;
        }
        if (lane == 0) {
            n_s = n;
            n_accepted[b] = n;
            next_token[b] = tgt_s[cur];
        }
    }
    __syncthreads();
    const int n = n_s, L = len_s;
    for (int i = tid; i < T; i += kThreads) accepted[(int64_t)b * T + i] = i < n ? path_s[i] : -1;
    const int64_t room = Lmax - L;
    const int nc = (int64_t)n < room ? n : (int)room;
    if (tid == 0 && nc < n) flag_error(dev_err, HTA_DEVERR_CACHE_LEN);
    // rows of d bf16 = d / 8 chunks of 16 bytes; K rows then V rows. Each
    // thread loads up to kBatch chunks before storing any, so a CTA keeps
    // kBatch x 256 loads in flight instead of one round trip per chunk.
    const int cpr = d / 8;
    const int per_kv = Hkv * nc * cpr;
    for (int base = tid; base < 2 * per_kv; base += kBatch * kThreads) {
        uint4 v[kBatch];
        int64_t dst[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int x = base + u * kThreads;
            dst[u] = -1;
            if (x < 2 * per_kv) {
                const int kv = x >= per_kv, y = x - kv * per_kv;
                const int h = y / (nc * cpr), r = y - h * nc * cpr, j = r / cpr, ch = r - j * cpr;
                const int64_t head = (int64_t)b * Hkv + h;
                if constexpr (!kGeneric) {
                    v[u] = (kv ? v_spec : k_spec)[(head * T + path_s[j]) * cpr + ch];
                    dst[u] = ((head * Lmax + L + j) * cpr + ch) * 2 + kv;  // chunk index, K/V in bit 0
                } else {
                    const int64_t src = st.nhd ? ((int64_t)b * T + path_s[j]) * Hkv + h : head * T + path_s[j];
                    const int64_t row = store_row(st, b, h, (int64_t)L + j, Hkv, Lmax);
                    if (row >= 0) {
                        v[u] = (kv ? v_spec : k_spec)[src * cpr + ch];
                        dst[u] = (row * cpr + ch) * 2 + kv;
                    } else if (ch == 0 && kv == 0) {
                        flag_error(dev_err, HTA_DEVERR_PAGE);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (dst[u] >= 0) ((dst[u] & 1) ? v_cache : k_cache)[dst[u] >> 1] = v[u];
    }
    __syncthreads();  // every thread has read cache_lens[b] (via len_s) before it changes
    if (tid == 0) cache_lens[b] = L + nc;
}

}  // namespace

cudaError_t accept_launch(const int32_t *parents, const int32_t *draft, const int32_t *target, int B, int T,
                          int Hkv, int d, int64_t Lmax, const void *k_spec, const void *v_spec, void *k_cache,
                          void *v_cache, int32_t *cache_lens, int32_t *accepted, int32_t *n_accepted,
                          int32_t *next_token, int32_t *dev_err, const KvStore &st, cudaStream_t stream) {
    if (st.nhd || st.page_size > 0)
        k_accept_commit<true><<<B, kThreads, 0, stream>>>(
            parents, draft, target, T, Hkv, d, Lmax, (const uint4 *)k_spec, (const uint4 *)v_spec, (uint4 *)k_cache,
            (uint4 *)v_cache, cache_lens, accepted, n_accepted, next_token, dev_err, st);
    else
        k_accept_commit<false><<<B, kThreads, 0, stream>>>(
            parents, draft, target, T, Hkv, d, Lmax, (const uint4 *)k_spec, (const uint4 *)v_spec, (uint4 *)k_cache,
            (uint4 *)v_cache, cache_lens, accepted, n_accepted, next_token, dev_err, st);
    return cudaGetLastError();
}

}  // namespace hta
