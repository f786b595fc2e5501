// Paired tcgen05 path of the hybrid tree attention: head dimension 128 and
// more than 128 packed query rows per KV head (T * G > 128).
//
// The method ("LongSpec: Long-Context Lossless Speculative Decoding with
// Efficient Drafting and Verification", Korean summary section 2.C, Dutch
// summary Methodologie section 3) splits the verification attention into an
// unmasked pass over the cached prefix and a masked pass over the tree tokens,
// merged by log-sum-exp; as in the single-CTA path, both passes are 128-key
// tiles of one persistent grid (all CTAs resident) and the cross-split merge runs
// after a grid barrier in the same launch.
//
// Here the grid is made of clusters of csize CTAs (2 to 4) on csize SMs. A
// cluster owns a range of tiles of the static split-KV schedule; a row group
// (up to csize x 128 packed rows of one KV head, whole tree nodes) is split
// into csize sub-groups of at most 128 rows, one per CTA. Each K/V tile is
// read from HBM once per cluster: CTA 0 loads the K tiles and CTA 1 the V
// tiles, each TMA copy multicast into every CTA's ring, and a ring stage is
// refilled only after the MMAs of every CTA have released it. With one
// 128-row sub-group per SM,
// tensor memory holds two S buffers next to O, so S(i+1) is computed while
// the softmax works on tile i and the softmax runs tile after tile:
//   warps 0, 3  TMA producers of the K ring and the V ring (CTA 0 issues the
//               K copies, CTA 1 the V copies, multicast to the cluster)
//   warp 1      MMA issuer: S(i) = Q K(i)^T into S[i % 2], O += P(i) V(i)
//   warp 2      TMA loads of each piece's Q rows (double-buffered)
//   warps 4-7   softmax, one query row per thread
// Tensor memory: S0 | S1 | O0 | O1, 128 columns each; P(i) (bf16) overwrites
// the first 64 columns of S[i % 2]; piece q accumulates into O[q % 2]. MMAs
// of one thread complete in issue order: S(0), S(1), then PV(i), S(i+2) for
// each tile, so S(i+2) never overwrites P(i) before PV(i) has read it.
// The softmax keeps the row max in base 2 (scores times scale * log2 e) and
// rescales O only when the max grows by more than 8 (factor 256); numerator
// and denominator share the stale max, so the result is exact.
// Every wait is bounded (~4e9 SM cycles); on expiry the kernel sets
// HTA_DEVERR_TIMEOUT and finishes instead of hanging.
#include <mutex>

#include "hta_launch.h"
#include "tc_host.h"
#include "tc_pipe.cuh"
#include "tc_ptx.cuh"

namespace hta {
namespace {

using namespace tc;
using namespace tcp;

constexpr int kTile = 128;                       // keys per tile
constexpr int kSubRows = 128;                    // query rows per CTA
constexpr int kThreads = 256;
constexpr uint32_t kTileBytes = 128 * 128 * 2;   // one K or V tile
constexpr uint32_t kSubBytes = 128 * 64 * 2;     // one 64-dim swizzled sub-tile of it
constexpr uint32_t kQBufBytes = kSubRows * 256;  // Q rows of one sub-group: two 64-dim sub-tiles
constexpr uint32_t kQSubBytes = kSubRows * 128;
constexpr int kMaxStages = 5;
constexpr uint32_t kOffQ = 0;                    // two Q buffers
constexpr uint32_t kOffRing = 2 * kQBufBytes;
constexpr uint32_t kSharedBytes = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;  // two O accumulators, alternating between pieces
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kMaxCluster = 4;                   // CTAs per cluster: 2 .. 4 (runtime)

// every CTA of this cluster, as a multicast mask
__device__ __forceinline__ uint16_t cluster_mask(const AttnParams &p) { return (uint16_t)((1u << p.csize) - 1u); }
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);

__host__ __device__ constexpr uint32_t off_shared(int stages) { return kOffRing + stages * kTileBytes; }
__host__ __device__ constexpr uint32_t off_sched(int stages) { return off_shared(stages) + kSharedBytes; }

struct Tc2Maps {
    CUtensorMap kc, vc, ks, vs, q;
};

struct Tc2Shared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];  // csize arrivals: the MMA warp of every CTA
    uint64_t s_full[2], p_full[2], pv_done[2], o_free[2], q_full[2], q_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
    int32_t arrived;  // the softmax warps have arrived on the grid barrier for this CTA
};
static_assert(sizeof(Tc2Shared) <= kSharedBytes, "shared control block too large");

// Rows of this CTA inside its row group: tree nodes [rank * tph, ...) of the
// group, all G heads of each (packed row t_local * G + g)
struct SubGroup {
    int32_t tpg, tph;  // tree nodes per group / per sub-group
    int32_t t0;        // first tree node of the sub-group inside the group
};

__device__ __forceinline__ SubGroup sub_group(const AttnParams &p, uint32_t rank) {
    SubGroup s;
    s.tpg = p.rows_pg / p.G;
    s.tph = (s.tpg + p.csize - 1) / p.csize;
    s.t0 = (int32_t)rank * s.tph;
    return s;
}

// ------------------------------------------------------------------ roles

// K tiles and V tiles stream through two rings of the same shared memory:
// K in stages [0, kKStages) and V in stages [kKStages, kStages). A K tile is
// released as soon as its S has been computed, a V tile only after its PV,
// so separate rings keep the K stream two tiles ahead of the MMAs. Stage
// and phase of tile j in each ring:
constexpr int kKStages = 2;
template <int kStages>
__device__ __forceinline__ uint32_t ring_stage(bool is_v, uint32_t j) {
    return is_v ? kKStages + j % (kStages - kKStages) : j % kKStages;
}
template <int kStages>
__device__ __forceinline__ uint32_t ring_round(bool is_v, uint32_t j) {
    return is_v ? j / (kStages - kKStages) : j / kKStages;
}

// One producer warp per ring. Every CTA expects the bytes of every tile on
// its own barrier; CTA 0 issues the K copies and CTA 1 the V copies, each
// multicast to every CTA of the cluster.
template <int kStages, bool kGeneric>
__device__ void producer(const AttnParams &p, const Tc2Maps &maps, Tc2Shared &sh, uint32_t ring, uint32_t rank,
                         bool is_v, const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const int n_tree = p.include_tree ? p.n_tree_tiles : 0;
    const int ring_n = is_v ? kStages - kKStages : kKStages;
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    uint32_t j = 0;  // tiles filled
    bool ok = true;
    const uint32_t leader = elect_one();
    const uint64_t policy = l2_evict_first_policy();  // K and V are read once
    [[maybe_unused]] PageWindow pw;  // paged layouts only
    while (ok && cursor_next(c, p, lens_s, pre_s, t)) {
        const bool tree = t.unit < n_tree;
        const int y = (tree ? t.unit : t.unit - n_tree) * kTile;
        const int z = t.b * p.Hkv + t.kvh;
        const uint32_t st = ring_stage<kStages>(is_v, j), round = ring_round<kStages>(is_v, j);
        // free in every CTA (and the previous round of full[st] is complete here)
        if (!wait_warp(bar_addr(sh.empty[st]), (round & 1) ^ 1, abort, p.dev_err)) {
            ok = false;
            break;
        }
        const uint32_t full = bar_addr(sh.full[st]);
        mbar_arrive_expect_tx_if(leader, full, kTileBytes);
        if ((uint32_t)is_v == rank) {
            const CUtensorMap *map = tree ? (is_v ? &maps.vs : &maps.ks) : (is_v ? &maps.vc : &maps.kc);
            if constexpr (!kGeneric) {
                // lanes 0 and 1 issue the two 64-dim halves in one instruction
                const uint32_t h = threadIdx.x & 1;
                tma_load_3d_mc_hint((threadIdx.x & 31) < 2 ? 1u : 0u, ring + st * kTileBytes + h * kSubBytes, map,
                                    full, (int)h * 64, y, z, cluster_mask(p), policy);
            } else {
                kv_tile_4d(p, pw, tree, t.b, t.kvh, y, t.Lb,
                           [&](bool on, uint32_t off, int c0, int c1, int c2, int c3) {
                               tma_load_4d_mc_hint(on ? 1u : 0u, ring + st * kTileBytes + off, map, full, c0, c1,
                                                   c2, c3, cluster_mask(p), policy);
                           });
            }
        }
        ++j;
    }
    if (!ok) {
        // let the copies already issued land before the CTA moves on
        const uint64_t t0 = cycles_now();
        for (uint32_t k = j > (uint32_t)ring_n ? j - ring_n : 0; k < j; ++k) {
            const uint32_t st = ring_stage<kStages>(is_v, k), round = ring_round<kStages>(is_v, k);
            while (!mbar_try_wait(bar_addr(sh.full[st]), round & 1))
                if (cycles_now() - t0 > kWaitLimitCycles) break;
        }
    }
}

// Q rows of this CTA's sub-group for each piece, into buffer q % 2: one box
// per 64-dim half, tph tree nodes x G heads, zero past the last tree node.
__device__ void q_loader(const AttnParams &p, const Tc2Maps &maps, Tc2Shared &sh, uint32_t sQ, uint32_t rank,
                         const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const uint32_t leader = elect_one();
    const SubGroup sg = sub_group(p, rank);
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    while (cursor_next(c, p, lens_s, pre_s, t)) {
        if (!t.first) continue;
        const uint32_t qb = t.q & 1;
        if (t.q >= 2 && !wait_warp(bar_addr(sh.q_empty[qb]), ((t.q - 2) >> 1) & 1, abort, p.dev_err)) return;
        const uint32_t full = bar_addr(sh.q_full[qb]);
        const int tq = t.rg * sg.tpg + sg.t0;
        mbar_arrive_expect_tx_if(leader, full, (uint32_t)(sg.tph * p.G) * 256u);
        tma_load_4d(leader, sQ + qb * kQBufBytes, &maps.q, full, 0, t.kvh * p.G, tq, t.b);
        tma_load_4d(leader, sQ + qb * kQBufBytes + kQSubBytes, &maps.q, full, 64, t.kvh * p.G, tq, t.b);
    }
}

// 8 MMAs over d = 128: S[128 x 128] = Q[128 x 128] K^T
__device__ __forceinline__ void issue_qk(uint32_t leader, uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t o = ((kk >> 2) * kSubBytes + (kk & 3) * 32) >> 4;  // same layout for Q and K
        mma_ss(leader, d_tmem, q_desc + o, k_desc + o, kIdescQK, kk > 0);
    }
}

// 8 MMAs over 128 keys: O[128 x 128] (+)= P[128 x 128] V[128 x 128]
__device__ __forceinline__ void issue_pv(uint32_t leader, uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(leader, o_tmem, p_tmem + kk * 8, v_desc + ((kk * 2048) >> 4), kIdescPV,
               (accumulate || kk > 0) ? 1u : 0u);
}

// S(j) into S[j % 2]: waits for K(j) and, at the start of a piece, for its
// Q rows; releases K(j) in every CTA and, after the last S of a piece, the
// piece's Q buffer
template <int kStages>
__device__ __forceinline__ bool issue_s(const AttnParams &p, Tc2Shared &sh, volatile int32_t *abort,
                                        uint32_t leader, uint32_t j, const TileInfo &t, uint32_t tmem,
                                        uint64_t q_desc0, uint64_t k_desc0) {
    const uint32_t st = ring_stage<kStages>(false, j), round = ring_round<kStages>(false, j);
    const uint32_t qb = t.q & 1;
    if (!wait_warp(bar_addr(sh.full[st]), round & 1, abort, p.dev_err)) return false;
    if (t.first && !wait_warp(bar_addr(sh.q_full[qb]), (t.q >> 1) & 1, abort, p.dev_err)) return false;
    tc_fence_after();
    issue_qk(leader, tmem + (j & 1) * 128, q_desc0 + ((qb * kQBufBytes) >> 4), k_desc0 + ((st * kTileBytes) >> 4));
    mma_commit(leader, bar_addr(sh.s_full[j & 1]));
    mma_commit_mc(leader, bar_addr(sh.empty[st]), cluster_mask(p));
    if (t.last) mma_commit(leader, bar_addr(sh.q_empty[qb]));
    return true;
}

template <int kStages>
__device__ void mma_issuer(const AttnParams &p, Tc2Shared &sh, uint32_t sQ, uint32_t ring, uint32_t tmem,
                           const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const uint32_t leader = elect_one();
    const uint64_t q_desc0 = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(ring, 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(ring, kSubBytes, 1024);
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo cur, n1, n2;
    if (!cursor_next(c, p, lens_s, pre_s, cur)) return;
    bool has1 = cursor_next(c, p, lens_s, pre_s, n1);
    bool has2 = has1 && cursor_next(c, p, lens_s, pre_s, n2);
    if (!issue_s<kStages>(p, sh, abort, leader, 0, cur, tmem, q_desc0, k_desc0)) return;
    if (has1 && !issue_s<kStages>(p, sh, abort, leader, 1, n1, tmem, q_desc0, k_desc0)) return;
    for (uint32_t i = 0;; ++i) {
        const uint32_t b = i & 1;
        const uint32_t stv = ring_stage<kStages>(true, i), rv = ring_round<kStages>(true, i);
        if (!wait_warp(bar_addr(sh.p_full[b]), (i >> 1) & 1, abort, p.dev_err)) return;
        if (!wait_warp(bar_addr(sh.full[stv]), rv & 1, abort, p.dev_err)) return;
        // O[q % 2] is free once the record of piece q - 2 has been read out
        if (cur.first && cur.q >= 2 &&
            !wait_warp(bar_addr(sh.o_free[cur.q & 1]), ((cur.q - 2) >> 1) & 1, abort, p.dev_err))
            return;
        tc_fence_after();
        issue_pv(leader, tmem + kColO + (cur.q & 1) * 128, tmem + b * 128, v_desc0 + ((stv * kTileBytes) >> 4),
                 !cur.first);
        mma_commit_mc(leader, bar_addr(sh.empty[stv]), cluster_mask(p));
        mma_commit(leader, bar_addr(sh.pv_done[b]));
        if (has2 && !issue_s<kStages>(p, sh, abort, leader, i + 2, n2, tmem, q_desc0, k_desc0)) return;
        if (!has1) break;
        cur = n1;
        n1 = n2;
        has1 = has2;
        has2 = has1 && cursor_next(c, p, lens_s, pre_s, n2);
    }
}

template <int kStages>
__device__ void softmax_wg(const AttnParams &p, Tc2Shared &sh, uint32_t ring, uint32_t tmem, uint32_t rank,
                           uint32_t worker, const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    griddep_wait();  // the mask build before this launch has finished
    volatile int32_t *abort = &sh.abort;
    const int lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;  // row of this sub-group == TMEM lane
    const int tid_wg = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int n_tree = p.include_tree ? p.n_tree_tiles : 0;
    const float c2 = p.scale_log2;
    const SubGroup sg = sub_group(p, rank);

    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    uint32_t gi = 0;
    float m_run = -INFINITY, l_run = 0.f;
    bool o_valid = false, valid = false;
    int r_group = 0;  // packed row inside the row group
    uint32_t mw[HTA_TMAX / 32], mw_next[HTA_TMAX / 32];
#pragma unroll
    for (int w = 0; w < HTA_TMAX / 32; ++w) mw[w] = mw_next[w] = 0u;
    // mask words of this thread's tree node in the piece starting at unit u
    // (loads issued early, consumed at that piece's first tile)
    auto load_mask = [&](int64_t u, uint32_t (&dst)[HTA_TMAX / 32]) {
        const UnitPos pos = locate_unit(p, u, lens_s, pre_s);
        const int nt = min(sg.tph, rows_in_group(p, pos.rg) / p.G - sg.t0);
        const bool v = row < nt * p.G;
        const int tn = v ? pos.rg * sg.tpg + (sg.t0 * p.G + row) / p.G : 0;
#pragma unroll
        for (int w = 0; w < HTA_TMAX / 32; ++w)
            dst[w] = (v && w < p.W) ? __ldg(p.mask + ((int64_t)pos.b * p.T + tn) * p.W + w) : 0u;
    };
    // A piece's record is written during the next piece, 32 columns after
    // each of its first tiles: the last PV of the piece has finished by then
    // (two O accumulators alternate between pieces), and the stores, which
    // queue behind the K/V stream, come in small batches instead of one
    // 64 KB burst that would stall the softmax.
    struct Pending {
        bool on, valid;
        int32_t r_group, k;  // next 32-column chunk
        uint32_t gi, ob;     // tile of the piece's last PV, O accumulator
        int64_t slot;
        float m, l;
    } pend = {false, false, 0, 0, 0, 0, 0, 0.f, 0.f};
    int pend_rows = 0;
    bool ok = true;
    auto write_record = [&](int chunks) -> bool {
        if (pend.k == 0) {
            if (!wait_warp(bar_addr(sh.pv_done[pend.gi & 1]), (pend.gi >> 1) & 1, abort, p.dev_err)) return false;
            tc_fence_after();
        }
        const uint32_t tOp = tmem + lane_off + kColO + pend.ob * 128;
        float *rec = p.ws_rec + (pend.slot * p.rows_pg + pend.r_group) * 132;
#pragma unroll 1
        for (int n = 0; n < chunks && pend.k < 4; ++n, ++pend.k) {
            uint32_t o[32];
            tmem_ld32(tOp + 32 * pend.k, o);
            if (pend.valid) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<uint4 *>(rec + 32 * pend.k + e) = make_uint4(o[e], o[e + 1], o[e + 2], o[e + 3]);
            }
        }
        if (pend.k == 4) {
            if (pend.valid) *reinterpret_cast<float2 *>(rec + 128) = make_float2(pend.m, pend.l);
            tc_fence_before();
            mbar_arrive(bar_addr(sh.o_free[pend.ob]));
            pend.on = false;
        }
        return true;
    };

    while (cursor_next(c, p, lens_s, pre_s, t)) {
        const uint32_t b = gi & 1;
        const uint32_t tS = tmem + lane_off + b * 128;
        const uint32_t tO = tmem + lane_off + kColO + (t.q & 1) * 128;
        if (t.first) {
            const int t_group = rows_in_group(p, t.rg) / p.G;  // tree nodes in this group
            const int nt = min(sg.tph, t_group - sg.t0);
            valid = row < nt * p.G;
            r_group = sg.t0 * p.G + row;
            if (p.include_tree) {
                if (t.q == 0) {
                    load_mask(c.u - (c.left + 1), mw);  // first piece: the unit of this tile
                } else {
#pragma unroll
                    for (int w = 0; w < HTA_TMAX / 32; ++w) mw[w] = mw_next[w];
                }
                // the next piece's words: global loads queue behind the K/V
                // stream for microseconds, so they are issued a piece ahead
                if (c.u < c.u_end) load_mask(c.u, mw_next);
            }
            m_run = -INFINITY;
            l_run = 0.f;
            o_valid = false;
        }
        const bool tree = t.unit < n_tree;
        const int j0 = (tree ? t.unit : t.unit - n_tree) * kTile;
        const int nvalid = tree ? min(kTile, p.T - j0) : min(kTile, t.Lb - j0);

        ok = wait_bar(bar_addr(sh.s_full[b]), (gi >> 1) & 1, abort, p.dev_err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        // a partial last cache tile: clear the V rows past the sequence end in
        // this CTA's copy (they may hold anything, and 0 * NaN would poison O)
        if (!tree && nvalid < kTile) {
            const uint32_t st = ring_stage<kStages>(true, gi), round = ring_round<kStages>(true, gi);
            ok = wait_bar(bar_addr(sh.full[st]), round & 1, abort, p.dev_err);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t vb = ring + st * kTileBytes;
            const int chunks = (kTile - nvalid) * 8;  // 16-byte chunks per sub-tile
            for (int ch = tid_wg; ch < 2 * chunks; ch += 128) {
                const int sub = ch / chunks, k = ch - sub * chunks;
                const uint32_t dst = vb + sub * kSubBytes + nvalid * 128 + k * 16;
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
            }
            fence_proxy_async_smem();
        }
        uint32_t sa[64], sb[64];  // raw scores of keys 0..63 and 64..127
        tmem_ld128(tS, sa, sb);
        // raw-score max (the scale is positive); masked keys become -inf
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
        if (!tree && nvalid == kTile) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
                mx[e & 7] = fmax3(mx[e & 7], __uint_as_float(sa[e]), __uint_as_float(sb[e]));
        } else {
            // the tree mask (a tree has at most two tiles of 128 keys; rows
            // past the sub-group see every key, their result is discarded)
            // and keys past the sequence end
            uint32_t w4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w4[k] = (tree && valid) ? (t.unit == 0 ? mw[k] : mw[4 + k]) : 0xffffffffu;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const bool va = e < nvalid && ((w4[e >> 5] >> (e & 31)) & 1u);
                const bool vb = (e + 64) < nvalid && ((w4[2 + (e >> 5)] >> (e & 31)) & 1u);
                if (!va) sa[e] = 0xff800000u;  // -inf
                if (!vb) sb[e] = 0xff800000u;
                mx[e & 7] = fmax3(mx[e & 7], __uint_as_float(sa[e]), __uint_as_float(sb[e]));
            }
        }
        const float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c2;
        // lazy rescale: the reference max moves only when the tile max passes
        // it by more than the threshold
        const float m_new = fmaxf(m_run, m_tile);
        const bool moved = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (moved) {
            alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
        }
        // P = 2^(s * scale * log2 e - m_run), packed to bf16 pairs over the first
        // 64 columns of this S buffer (all of S is already in registers), in
        // 16-column chunks stored as soon as each is complete
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float x0, x1;  // score pairs through the packed fp32 unit
                fma2(x0, x1, __uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1]), c2, neg_m);
                const float p0 = ex2(x0), p1 = ex2(x1);
                add2(ls[2 * (e & 1)], ls[2 * (e & 1) + 1], p0, p1);
                pk[e] = pack_bf16x2(p0, p1);
                if (e == 15) tmem_st16(tS, pk);
            }
            tmem_st16(tS + 16, pk + 16);
        }
        {
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float x0, x1;  // score pairs through the packed fp32 unit
                fma2(x0, x1, __uint_as_float(sb[2 * e]), __uint_as_float(sb[2 * e + 1]), c2, neg_m);
                const float p0 = ex2(x0), p1 = ex2(x1);
                add2(ls[2 * (e & 1)], ls[2 * (e & 1) + 1], p0, p1);
                pk[e] = pack_bf16x2(p0, p1);
                if (e == 15) tmem_st16(tS + 32, pk);
            }
            tmem_st16(tS + 32 + 16, pk + 16);
        }
        if (__any_sync(0xffffffffu, moved && o_valid)) {
            // O is stable once PV of the previous tile has finished (PV of
            // this tile cannot start before this warpgroup's P)
            ok = wait_bar(bar_addr(sh.pv_done[(gi - 1) & 1]), ((gi - 1) >> 1) & 1, abort, p.dev_err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const float a = (moved && o_valid) ? alpha : 1.f;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * k, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                tmem_st32(tO + 32 * k, o);
            }
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_addr(sh.p_full[b]));
        o_valid = true;

        // a part of the previous piece's record (all of what is left of it at
        // the end of a piece of fewer than four tiles)
        if (pend.on && !write_record(t.last ? 4 : 1)) break;
        if (t.last) {
            pend = {true, valid, r_group, 0, gi, (uint32_t)(t.q & 1), slot_of(p, t.seg, worker), m_run, l_run};
            pend_rows = max(0, min(sg.tph, rows_in_group(p, t.rg) / p.G - sg.t0)) * p.G;
        }
        ++gi;
    }
    // The last piece's record: rows staged in shared memory (the ring is idle:
    // every tile of this CTA has landed and been consumed), written with one
    // bulk store, after which this CTA arrives on the grid barrier. Every
    // softmax thread reaches the named barrier once, whatever happened before;
    // a timeout anywhere (abort set) leaves the arrival to the merge phase.
    bool rec = pend.on && ok && *abort == 0;
    if (rec) {
        rec = wait_bar(bar_addr(sh.pv_done[pend.gi & 1]), (pend.gi >> 1) & 1, abort, p.dev_err);
        if (__all_sync(0xffffffffu, rec)) {
            tc_fence_after();
            const uint32_t tOp = tmem + lane_off + kColO + pend.ob * 128;
            const uint32_t srow = ring + (uint32_t)row * 528u;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                uint32_t o[32];
                tmem_ld32(tOp + 32 * k, o);
#pragma unroll
                for (int e = 0; e < 32; e += 4) sts_v4(srow + (uint32_t)(32 * k + e) * 4u, o[e], o[e + 1], o[e + 2], o[e + 3]);
            }
            sts_v2(srow + 512u, pend.m, pend.l);
            fence_proxy_async_smem();
        }
    }
    named_sync(1, 128);
    if (tid_wg == 0 && pend.on && *abort == 0) {
        if (pend_rows > 0)
            bulk_store(p.ws_rec + (pend.slot * p.rows_pg + sg.t0 * p.G) * 132, ring, (uint32_t)pend_rows * 528u);
        bulk_store_commit_and_wait();
        fence_proxy_async_all();
        __threadfence();
        atomicAdd(&p.bar[0], 1u);
        sh.arrived = 1;
    }
}

// kGeneric: K/V stored in any layout but contiguous head-major (4-D maps,
// paged pools). kCS: CTAs per cluster, fixed at compile time so that the
// cluster shape is part of the kernel itself and every launch of it, by any
// launcher, runs as clusters of kCS CTAs.
template <int kStages, bool kGeneric, int kCS>
__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kThreads, 1)
    k_tc2_verify(const __grid_constant__ AttnParams p, const __grid_constant__ Tc2Maps maps) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned (128-byte swizzle atoms), by pointer arithmetic on the
    // shared array so that accesses through it stay shared-memory accesses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Tc2Shared &sh = *reinterpret_cast<Tc2Shared *>(smem + off_shared(kStages));
    int32_t *lens_s = reinterpret_cast<int32_t *>(smem + off_sched(kStages));
    int64_t *pre_s = reinterpret_cast<int64_t *>(smem + off_sched(kStages) + ((p.B * 4 + 15) / 16) * 16);
    int64_t *lo_s = pre_s + p.B + 1;
    const uint32_t sQ = smem_u32(smem + kOffQ), ring = smem_u32(smem + kOffRing);
    const int warp = threadIdx.x >> 5;
    // Every cluster operation below (multicast copies and commits, cluster
    // barriers) assumes a cluster of exactly csize CTAs and one worker per
    // cluster; a launch in any other shape writes nothing and says so.
    if (p.csize != kCS || cluster_nctarank() != (uint32_t)kCS || gridDim.x != (uint32_t)kCS * (uint32_t)p.workers) {
        if (threadIdx.x == 0) flag_error(p.dev_err, HTA_DEVERR_LAUNCH);
        return;
    }
    const uint32_t rank = cluster_ctarank(), worker = cluster_id_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_addr(sh.full[s]), 1);
            mbar_init(bar_addr(sh.empty[s]), (uint32_t)p.csize);  // the MMA warp of every CTA
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(sh.s_full[b]), 1);
            mbar_init(bar_addr(sh.p_full[b]), 128);
            mbar_init(bar_addr(sh.q_full[b]), 1);
            mbar_init(bar_addr(sh.q_empty[b]), 1);
            mbar_init(bar_addr(sh.pv_done[b]), 1);
        }
        mbar_init(bar_addr(sh.o_free[0]), 128);
        mbar_init(bar_addr(sh.o_free[1]), 128);
        mbar_init(bar_addr(sh.drain), 1);
        sh.abort = 0;
        sh.arrived = 0;
        mbar_fence_init();
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.kc);
        tma_prefetch_desc(&maps.vc);
        if (p.include_tree) {
            tma_prefetch_desc(&maps.ks);
            tma_prefetch_desc(&maps.vs);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // every CTA's barriers exist before any multicasts into another: the
    // cluster barrier's round trip overlaps the schedule below
    cluster_arrive();
    // The only kernel that lets this one start before it has finished is the
    // mask build, which writes the tree mask alone and lets it start only
    // once every kernel before the mask build has finished: the softmax warps,
    // which read the mask, wait for it; everything else starts at once
    build_schedule(p, lens_s, pre_s, lo_s);  // ends with __syncthreads
    cluster_wait();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t u0 = lo_s[worker], u1 = lo_s[worker + 1];

    if (warp == 0 || warp == 3)
        producer<kStages, kGeneric>(p, maps, sh, ring, rank, warp == 3, lens_s, pre_s, u0, u1);
    else if (warp == 1)
        mma_issuer<kStages>(p, sh, sQ, ring, tmem, lens_s, pre_s, u0, u1);
    else if (warp == 2)
        q_loader(p, maps, sh, sQ, rank, lens_s, pre_s, u0, u1);
    else if (warp >= 4)
        softmax_wg<kStages>(p, sh, ring, tmem, rank, worker, lens_s, pre_s, u0, u1);
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        // every MMA of this CTA has finished before tensor memory is freed
        mma_commit(elect_one(), bar_addr(sh.drain));
        const uint64_t t0 = cycles_now();
        while (!mbar_try_wait(bar_addr(sh.drain), 0))
            if (cycles_now() - t0 > kWaitLimitCycles) break;
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // Every multicast fill of this CTA's ring has landed (its own waits saw
    // each tile), so Q and the ring are idle now and stage the merge; the
    // peers' last releases may still arrive on this CTA's ring barriers,
    // outside that region, so the CTA leaves only after every CTA of the
    // cluster has come this far
    cluster_arrive();
    merge_phase<128, 12>(p, lens_s, pre_s, lo_s, smem + kOffQ, sh.arrived != 0);  // 12 records per round trip
    grid_barrier_depart(p);
    cluster_wait();
}

size_t tc2_smem_bytes(int stages, int B, int workers) {
    return 1024 + off_sched(stages) + sched_bytes(B, workers);
}

int tc2_stages(int B, int workers) {
    int max_smem = 0, dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    const size_t slack = 256;  // static shared memory of the merge and barrier helpers
    if (tc2_smem_bytes(5, B, workers) + slack <= (size_t)max_smem) return 5;
    if (tc2_smem_bytes(4, B, workers) + slack <= (size_t)max_smem) return 4;
    return 0;
}

// The cluster shape comes from the kernel's compile-time cluster dimensions;
// the launch adds programmatic serialization (and a cooperative grid when
// requested: the merge waits on every CTA, see cooperative_requested).
template <int kStages, bool kGeneric, int kCS>
cudaError_t launch_cs(const AttnParams &p, const Tc2Maps &maps, int grid, cudaStream_t stream) {
    const size_t smem = tc2_smem_bytes(kStages, p.B, grid / kCS);
    cudaError_t e = cudaFuncSetAttribute(k_tc2_verify<kStages, kGeneric, kCS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cooperative_requested()) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n++].val.cooperative = 1;
    }
    return launch_dependent(cfg, attr, n, k_tc2_verify<kStages, kGeneric, kCS>, p, maps);
}

template <int kStages, bool kGeneric>
cudaError_t launch_stages(const AttnParams &p, const Tc2Maps &maps, int grid, cudaStream_t stream) {
    switch (p.csize) {
        case 2: return launch_cs<kStages, kGeneric, 2>(p, maps, grid, stream);
        case 3: return launch_cs<kStages, kGeneric, 3>(p, maps, grid, stream);
        case 4: return launch_cs<kStages, kGeneric, 4>(p, maps, grid, stream);
    }
    return cudaErrorInvalidValue;
}

template <int kStages, int kCS>
int max_clusters_cs(int B, int num_sms) {
    const size_t smem = tc2_smem_bytes(kStages, B, num_sms / 2);
    if (cudaFuncSetAttribute(k_tc2_verify<kStages, false, kCS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((num_sms / kCS) * kCS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)k_tc2_verify<kStages, false, kCS>, &cfg) != cudaSuccess) return 0;
    return n;
}

template <int kStages>
int max_clusters(int B, int num_sms, int csize) {
    switch (csize) {
        case 2: return max_clusters_cs<kStages, 2>(B, num_sms);
        case 3: return max_clusters_cs<kStages, 3>(B, num_sms);
        case 4: return max_clusters_cs<kStages, 4>(B, num_sms);
    }
    return 0;
}

}  // namespace

int tc2_tile() { return kTile; }
int tc2_rows_per_sub() { return kSubRows; }

// CTAs of the largest co-resident grid of csize-CTA clusters (0 if none); the
// occupancy query runs once per device, ring depth and cluster size
int tc2_max_grid(int B, int num_sms, int csize) {
    if (csize < 2 || csize > kMaxCluster) return 0;
    const int stages = tc2_stages(B, num_sms / 2);
    if (stages == 0) return 0;
    static std::mutex mu;
    static int cached[64][2][kMaxCluster + 1];  // [device][stages == 5][csize], 0 = not yet queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int &n = cached[dev][stages == 5 ? 1 : 0][csize];
    if (n == 0) n = 1 + (stages == 5 ? max_clusters<5>(B, num_sms, csize) : max_clusters<4>(B, num_sms, csize));
    const int clusters = n - 1;
    return csize * (clusters < num_sms / csize ? clusters : num_sms / csize);
}

cudaError_t tc2_launch(const AttnParams &p, int grid, cudaStream_t stream) {
    Tc2Maps maps;
    memset(&maps, 0, sizeof maps);
    const int64_t heads = (int64_t)p.B * p.Hkv;
    if (p.csize < 2 || p.csize > kMaxCluster || grid < p.csize || grid % p.csize != 0 || p.workers != grid / p.csize)
        return cudaErrorInvalidValue;
    // row groups of whole tree nodes, each half at most 128 rows
    if (p.G < 1 || p.rows_pg % p.G != 0) return cudaErrorInvalidValue;
    const int tpg = p.rows_pg / p.G, tph = (tpg + p.csize - 1) / p.csize;
    if (tph * p.G > kSubRows) return cudaErrorInvalidValue;
    if (!tch::encode_q(&maps.q, p.q, p.B, p.T, p.Hq, p.G, tph)) return cudaErrorInvalidValue;
    if (!tch::encode_kv_maps(p, heads, kTile, &maps.kc, &maps.vc, &maps.ks, &maps.vs)) return cudaErrorInvalidValue;
    const int stages = tc2_stages(p.B, grid / p.csize);
    if (stages == 5)
        return p.kv_generic ? launch_stages<5, true>(p, maps, grid, stream)
                            : launch_stages<5, false>(p, maps, grid, stream);
    if (stages == 4)
        return p.kv_generic ? launch_stages<4, true>(p, maps, grid, stream)
                            : launch_stages<4, false>(p, maps, grid, stream);
    return cudaErrorInvalidConfiguration;
}

}  // namespace hta
