// tcgen05 tensor-core path of the hybrid tree attention (head dimension 128).
//
// The method ("LongSpec: Long-Context Lossless Speculative Decoding with
// Efficient Drafting and Verification", Korean summary section 2.C, Dutch
// summary Methodologie section 3) splits the verification attention into an
// unmasked pass over the long cached prefix and a masked pass over the tree
// tokens, merged by log-sum-exp. Here both passes are 128-key tiles of one
// persistent grid (one CTA per SM, all resident, a static split-KV schedule
// balanced by tile count, see hta_internal.cuh), and the cross-split and
// cross-part merge runs after a grid barrier in the same launch.
//
// One CTA works on a row group of up to 256 packed query rows of one KV head
// (row r = t*G + g, so every K/V tile is shared by all G query heads of the
// tree), as two 128-row halves:
//   warp 0        TMA producer: K and V tiles (128 keys x 128 dims, bf16,
//                 128-byte swizzle) into a shared-memory ring;
//   warp 1        MMA issuer: S_h = Q_h K(i)^T into tensor memory, then
//                 O_h += P_h V(i) with P read from tensor memory;
//   warp 2        TMA loads of each piece's Q rows (both halves at once);
//   warps 4-7     softmax of half 0, one query row per thread;
//   warps 8-11    softmax of half 1.
// Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1, 128 columns each; P_h
// (bf16) overwrites the first 64 columns of S_h. The MMA warp issues
// PV(0,i), S(0,i+1), PV(1,i), S(1,i+1): while the softmax of one half works,
// the tensor core runs the other half's products. Tensor-core operations of
// one thread execute in issue order, so S(h,i+1) never overtakes PV(h,i)
// that still reads P_h, and the arrival of S(h,i) implies PV(h,i-1) is done
// (the softmax may then rescale O_h). The softmax keeps the row max in base 2
// (scores times scale*log2 e) and rescales O only when the max grows by more
// than 8 (factor 256); numerator and denominator share the stale max, so the
// result is exact.
//
// Producer and MMA warps run their loops warp-uniformly; one elected lane
// issues each TMA / MMA / commit. Every wait is bounded (~4e9 SM cycles,
// about 2 s); on expiry the kernel sets HTA_DEVERR_TIMEOUT, waits for its own
// copies in flight, frees its tensor memory and finishes instead of hanging.
#include "hta_launch.h"
#include "tc_host.h"
#include "tc_pipe.cuh"
#include "tc_ptx.cuh"

namespace hta {
namespace {

using namespace tc;
using namespace tcp;

constexpr int kTile = 128;          // keys per tile
constexpr int kHalf = 128;          // query rows per MMA
constexpr int kMaxRows = 256;       // rows per row group
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = 128 * 128 * 2;   // one K or V tile
constexpr uint32_t kSubBytes = 128 * 64 * 2;     // one 64-dim swizzled sub-tile of it
constexpr uint32_t kQSubBytes = kMaxRows * 64 * 2;  // 64 dims of all rows of a group
constexpr uint32_t kQHalfBytes = kHalf * 128;       // offset of half h inside a sub-tile
constexpr int kMaxStages = 5;                    // K/V ring stages (4 when the schedule is large)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = 2 * kQSubBytes;
constexpr uint32_t kSharedBytes = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;  // S_0, S_1 take columns 0..255
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);

__host__ __device__ constexpr uint32_t off_shared(int stages) { return kOffRing + stages * kTileBytes; }
__host__ __device__ constexpr uint32_t off_sched(int stages) { return off_shared(stages) + kSharedBytes; }

struct TcMaps {
    CUtensorMap kc, vc, ks, vs, q;
};

struct TcShared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2], q_full, q_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(TcShared) <= kSharedBytes, "shared control block too large");

// ------------------------------------------------------------------ roles

template <int kStages, bool kGeneric>
__device__ void producer(const AttnParams &p, const TcMaps &maps, TcShared &sh, uint32_t ring,
                         const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const int n_tree = p.include_tree ? p.n_tree_tiles : 0;
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    uint32_t n = 0;  // ring fills issued
    bool ok = true;
    const uint32_t leader = elect_one();
    // K and V are streamed once: keep them from evicting everything else in L2
    const uint64_t policy = l2_evict_first_policy();
    [[maybe_unused]] PageWindow pw;  // paged layouts only
    while (ok && cursor_next(c, p, lens_s, pre_s, t)) {
        const bool tree = t.unit < n_tree;
        const int y = (tree ? t.unit : t.unit - n_tree) * kTile;
        const int z = t.b * p.Hkv + t.kvh;
        for (int kv = 0; kv < 2; ++kv, ++n) {
            const uint32_t st = n % kStages, round = n / kStages;
            if (!wait_warp(bar_addr(sh.empty[st]), (round & 1) ^ 1, abort, p.dev_err)) {
                ok = false;
                break;
            }
            const CUtensorMap *map = tree ? (kv ? &maps.vs : &maps.ks) : (kv ? &maps.vc : &maps.kc);
            const uint32_t full = bar_addr(sh.full[st]);
            mbar_arrive_expect_tx_if(leader, full, kTileBytes);
            if constexpr (!kGeneric) {
                // lanes 0 and 1 issue the two 64-dim halves in one instruction
                const uint32_t h = threadIdx.x & 1;
                tma_load_3d_hint((threadIdx.x & 31) < 2 ? 1u : 0u, ring + st * kTileBytes + h * kSubBytes, map, full,
                                 (int)h * 64, y, z, policy);
            } else {
                kv_tile_4d(p, pw, tree, t.b, t.kvh, y, t.Lb,
                           [&](bool on, uint32_t off, int c0, int c1, int c2, int c3) {
                               tma_load_4d_hint(on ? 1u : 0u, ring + st * kTileBytes + off, map, full, c0, c1, c2,
                                                c3, policy);
                           });
            }
        }
    }
    if (!ok) {
        // let the copies already issued land before the CTA exits
        const uint64_t t0 = cycles_now();
        for (uint32_t k = n > (uint32_t)kStages ? n - kStages : 0; k < n; ++k) {
            const uint32_t st = k % kStages, round = k / kStages;
            while (!mbar_try_wait(bar_addr(sh.full[st]), round & 1))
                if (cycles_now() - t0 > kWaitLimitCycles) break;
        }
    }
}

// Q rows of each piece's row group, by TMA: one box per 64-dim half covering
// every (tree node, query head) of the group, 128-byte swizzled, zero past
// the last tree node. The group's rows are t-aligned (rows_pg = tpg * G), so
// box row t_local * G + g is packed row r_local. A piece's Q replaces the
// previous one only after the MMAs of that piece have read it (q_empty).
__device__ void q_loader(const AttnParams &p, const TcMaps &maps, TcShared &sh, uint32_t sQ,
                         const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const uint32_t leader = elect_one();
    const int tpg = p.rows_pg / p.G;
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    while (cursor_next(c, p, lens_s, pre_s, t)) {
        if (!t.first) continue;
        if (t.q > 0 && !wait_warp(bar_addr(sh.q_empty), (t.q - 1) & 1, abort, p.dev_err)) return;
        const uint32_t full = bar_addr(sh.q_full);
        mbar_arrive_expect_tx_if(leader, full, (uint32_t)p.rows_pg * 256u);
        tma_load_4d(leader, sQ, &maps.q, full, 0, t.kvh * p.G, t.rg * tpg, t.b);
        tma_load_4d(leader, sQ + kQSubBytes, &maps.q, full, 64, t.kvh * p.G, t.rg * tpg, t.b);
    }
}

// 8 MMAs over d = 128: S_h[128 x 128] = Q_h[128 x 128] K^T
__device__ __forceinline__ void issue_qk(uint32_t leader, uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t qo = ((kk >> 2) * kQSubBytes + (kk & 3) * 32) >> 4;
        const uint32_t ko = ((kk >> 2) * kSubBytes + (kk & 3) * 32) >> 4;
        mma_ss(leader, d_tmem, q_desc + qo, k_desc + ko, kIdescQK, kk > 0);
    }
}

// 8 MMAs over 128 keys: O_h[128 x 128] (+)= P_h[128 x 128] V[128 x 128]
__device__ __forceinline__ void issue_pv(uint32_t leader, uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(leader, o_tmem, p_tmem + kk * 8, v_desc + ((kk * 2048) >> 4), kIdescPV,
               (accumulate || kk > 0) ? 1u : 0u);
}

// S(h,j): waits for K(j) (on the first half) and, at the start of a piece,
// for the group's Q rows; the last S of a piece releases Q
template <int kStages>
__device__ __forceinline__ bool issue_s_tile(const AttnParams &p, TcShared &sh, volatile int32_t *abort,
                                             uint32_t leader, int h, int halves, uint32_t j, const TileInfo &t,
                                             uint32_t tmem, uint64_t q_desc0, uint64_t k_desc0) {
    const uint32_t n = 2 * j, st = n % kStages, round = n / kStages;
    if (h == 0 && !wait_warp(bar_addr(sh.full[st]), round & 1, abort, p.dev_err)) return false;
    if (t.first && h == 0 && !wait_warp(bar_addr(sh.q_full), t.q & 1, abort, p.dev_err)) return false;
    tc_fence_after();
    issue_qk(leader, tmem + h * 128, q_desc0 + ((h * kQHalfBytes) >> 4), k_desc0 + ((st * kTileBytes) >> 4));
    mma_commit(leader, bar_addr(sh.s_full[h]));
    if (h == halves - 1) {
        mma_commit(leader, bar_addr(sh.empty[st]));
        if (t.last) mma_commit(leader, bar_addr(sh.q_empty));
    }
    return true;
}

// Issue order: S(0,0), S(1,0), then per tile i: PV(0,i), S(0,i+1), PV(1,i),
// S(1,i+1). The first S of a piece waits for the piece's Q rows; the first
// PV of a piece waits until the softmax has read out the previous piece's O.
template <int kStages>
__device__ void mma_issuer(const AttnParams &p, TcShared &sh, uint32_t sQ, uint32_t ring, uint32_t tmem,
                           int halves, const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    volatile int32_t *abort = &sh.abort;
    const uint32_t leader = elect_one();
    const uint64_t q_desc0 = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(ring, 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(ring, kSubBytes, 1024);
    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo cur, nxt;
    if (!cursor_next(c, p, lens_s, pre_s, cur)) return;
    bool has_next = cursor_next(c, p, lens_s, pre_s, nxt);

    for (int h = 0; h < halves; ++h)
        if (!issue_s_tile<kStages>(p, sh, abort, leader, h, halves, 0, cur, tmem, q_desc0, k_desc0)) return;
    for (uint32_t i = 0;; ++i) {
        const uint32_t nv = 2 * i + 1, stv = nv % kStages, rv = nv / kStages;
        if (!wait_warp(bar_addr(sh.full[stv]), rv & 1, abort, p.dev_err)) return;
        const uint64_t v_desc = v_desc0 + ((stv * kTileBytes) >> 4);
        for (int h = 0; h < halves; ++h) {
            if (!wait_warp(bar_addr(sh.p_full[h]), i & 1, abort, p.dev_err)) return;
            if (cur.first && cur.q > 0 && !wait_warp(bar_addr(sh.o_free[h]), (cur.q - 1) & 1, abort, p.dev_err))
                return;
            tc_fence_after();
            issue_pv(leader, tmem + kColO + h * 128, tmem + h * 128, v_desc, !cur.first);
            if (h == halves - 1) mma_commit(leader, bar_addr(sh.empty[stv]));
            if (cur.last) mma_commit(leader, bar_addr(sh.o_done[h]));
            if (has_next && !issue_s_tile<kStages>(p, sh, abort, leader, h, halves, i + 1, nxt, tmem, q_desc0, k_desc0))
                return;
        }
        if (!has_next) break;
        cur = nxt;
        has_next = cursor_next(c, p, lens_s, pre_s, nxt);
    }
}

template <int kStages>
__device__ void softmax_wg(const AttnParams &p, TcShared &sh, uint32_t ring, uint32_t tmem,
                           int h, const int32_t *lens_s, const int64_t *pre_s, int64_t u0, int64_t u1) {
    griddep_wait();  // the mask build before this launch has finished
    volatile int32_t *abort = &sh.abort;
    const int lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) & 3;
    const int row = wq * 32 + lane;  // row of this half == TMEM lane
    const int tid_wg = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + h * 128;
    const uint32_t tO = tmem + lane_off + kColO + h * 128;
    const int n_tree = p.include_tree ? p.n_tree_tiles : 0;
    const float c2 = p.scale_log2;

    Cursor c;
    cursor_init(c, u0, u1);
    TileInfo t;
    uint32_t gi = 0;
    float m_run = -INFINITY, l_run = 0.f;
    bool o_valid = false, valid = false;
    int r_local = 0;
    uint32_t mw[HTA_TMAX / 32];
#pragma unroll
    for (int w = 0; w < HTA_TMAX / 32; ++w) mw[w] = 0u;

    while (cursor_next(c, p, lens_s, pre_s, t)) {
        if (t.first) {
            const int nrows = rows_in_group(p, t.rg);
            r_local = h * kHalf + row;
            valid = r_local < nrows;
            const int r = t.rg * p.rows_pg + r_local;
            const int tn = valid ? r / p.G : 0;
            if (p.include_tree) {
#pragma unroll
                for (int w = 0; w < HTA_TMAX / 32; ++w)
                    mw[w] = (valid && w < p.W) ? __ldg(p.mask + ((int64_t)t.b * p.T + tn) * p.W + w) : 0u;
            }
            m_run = -INFINITY;
            l_run = 0.f;
            o_valid = false;
        }
        const bool tree = t.unit < n_tree;
        const int j0 = (tree ? t.unit : t.unit - n_tree) * kTile;
        const int nvalid = tree ? min(kTile, p.T - j0) : min(kTile, t.Lb - j0);

        bool ok = wait_bar(bar_addr(sh.s_full[h]), gi & 1, abort, p.dev_err);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
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
            // mask words of this tile (a tree has at most two tiles of 128
            // keys); rows past the group see every key (their result is
            // discarded)
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
        const float m_new = fmaxf(m_run, m_tile);
        const bool need = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
            alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
        }
        if (__any_sync(0xffffffffu, need && o_valid)) {
            // S_h arrived after PV(h, previous tile) finished: O_h is stable
            const float a = (need && o_valid) ? alpha : 1.f;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * k, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                tmem_st32(tO + 32 * k, o);
            }
            tmem_wait_st();
        }
        // a partial last cache tile: clear the V rows past the sequence end
        // (they may hold anything, and 0 * NaN would poison O)
        if (h == 0 && !tree && nvalid < kTile) {
            const uint32_t n = 2 * gi + 1, st = n % kStages, round = n / kStages;
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
        // P = 2^(s * scale * log2 e - m), packed to bf16 pairs over the first
        // 64 columns of S_h (all of S_h is already in registers)
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
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_addr(sh.p_full[h]));
        o_valid = true;

        if (t.last) {
            ok = wait_bar(bar_addr(sh.o_done[h]), t.q & 1, abort, p.dev_err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            float *rec = p.ws_rec + (slot_of(p, t.seg, blockIdx.x) * p.rows_pg + r_local) * 132;
#pragma unroll 1
            for (int k = 0; k < 4; ++k) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * k, o);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<uint4 *>(rec + 32 * k + e) = make_uint4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                }
            }
            if (valid) *reinterpret_cast<float2 *>(rec + 128) = make_float2(m_run, l_run);
            tc_fence_before();
            mbar_arrive(bar_addr(sh.o_free[h]));
        }
        ++gi;
    }
}

// kGeneric: K/V stored in any layout but contiguous head-major (4-D maps,
// paged pools)
template <int kStages, bool kGeneric = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_verify(const __grid_constant__ AttnParams p, const __grid_constant__ TcMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned (128-byte swizzle atoms), by pointer arithmetic on the
    // shared array so that accesses through it stay shared-memory accesses
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    TcShared &sh = *reinterpret_cast<TcShared *>(smem + off_shared(kStages));
    int32_t *lens_s = reinterpret_cast<int32_t *>(smem + off_sched(kStages));
    int64_t *pre_s = reinterpret_cast<int64_t *>(smem + off_sched(kStages) + ((p.B * 4 + 15) / 16) * 16);
    int64_t *lo_s = pre_s + p.B + 1;
    const uint32_t sQ = smem_u32(smem + kOffQ), ring = smem_u32(smem + kOffRing);
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_addr(sh.full[s]), 1);
            mbar_init(bar_addr(sh.empty[s]), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar_addr(sh.s_full[h]), 1);
            mbar_init(bar_addr(sh.p_full[h]), 128);
            mbar_init(bar_addr(sh.o_done[h]), 1);
            mbar_init(bar_addr(sh.o_free[h]), 128);
        }
        mbar_init(bar_addr(sh.q_full), 1);
        mbar_init(bar_addr(sh.q_empty), 1);
        mbar_init(bar_addr(sh.drain), 1);
        sh.abort = 0;
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
    // The only kernel that lets this one start before it has finished is the
    // mask build, which writes the tree mask alone and lets it start only
    // once every kernel before the mask build has finished: the softmax warps,
    // which read the mask, wait for it; everything else starts at once
    build_schedule(p, lens_s, pre_s, lo_s);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int64_t u0 = lo_s[blockIdx.x], u1 = lo_s[blockIdx.x + 1];
    const int halves = (p.rows_pg + kHalf - 1) / kHalf;

    // register split: 128 x 88 for the control warpgroup, 256 x 208 for the
    // softmax warpgroups (= 384 x 168 at launch); restored before the merge
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
        if (warp == 0)
            producer<kStages, kGeneric>(p, maps, sh, ring, lens_s, pre_s, u0, u1);
        else if (warp == 1)
            mma_issuer<kStages>(p, sh, sQ, ring, tmem, halves, lens_s, pre_s, u0, u1);
        else if (warp == 2)
            q_loader(p, maps, sh, sQ, lens_s, pre_s, u0, u1);
        __syncwarp();
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 208;");
        const int h = (warp >> 2) - 1;
        if (h < halves) softmax_wg<kStages>(p, sh, ring, tmem, h, lens_s, pre_s, u0, u1);
        __syncwarp();
        asm volatile("setmaxnreg.dec.sync.aligned.u32 168;");
    }
    __syncthreads();
    if (warp < 4) asm volatile("setmaxnreg.inc.sync.aligned.u32 168;");
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
    // Q and the K/V ring are idle now: they stage the merge
    merge_phase<128, 2>(p, lens_s, pre_s, lo_s, smem + kOffQ);  // 2 records per round trip: the register budget of 384 threads
    grid_barrier_depart(p);
}

size_t tc_smem_bytes(int stages, int B, int grid) {
    return 1024 + off_sched(stages) + sched_bytes(B, grid);
}

// Deepest ring that fits next to the schedule arrays of this batch
int tc_stages(int B, int grid) {
    int max_smem = 0, dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    // static shared memory of the merge and barrier helpers
    const size_t slack = 256;
    if (tc_smem_bytes(5, B, grid) + slack <= (size_t)max_smem) return 5;
    if (tc_smem_bytes(4, B, grid) + slack <= (size_t)max_smem) return 4;
    return 0;
}

template <int kStages, bool kGeneric>
cudaError_t launch_stages(const AttnParams &p, const TcMaps &maps, int grid, cudaStream_t stream) {
    const size_t smem = tc_smem_bytes(kStages, p.B, grid);
    cudaError_t e = cudaFuncSetAttribute(k_tc_verify<kStages, kGeneric>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
    return launch_dependent(cfg, attr, n, k_tc_verify<kStages, kGeneric>, p, maps);
}

}  // namespace

int tc_rows_per_group() { return kMaxRows; }
int tc_tile() { return kTile; }

int tc_max_grid(int B, int num_sms) {
    const int stages = tc_stages(B, num_sms);
    if (stages == 0) return 0;
    const size_t smem = tc_smem_bytes(stages, B, num_sms);
    int occ = 0;
    if (stages == 5) {
        if (cudaFuncSetAttribute(k_tc_verify<5>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_tc_verify<5>, kThreads, smem) != cudaSuccess)
            return 0;
    } else {
        if (cudaFuncSetAttribute(k_tc_verify<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_tc_verify<4>, kThreads, smem) != cudaSuccess)
            return 0;
    }
    return occ >= 1 ? num_sms : 0;  // one CTA per SM (the boundary table is sized for that)
}

cudaError_t tc_launch(const AttnParams &p, int grid, cudaStream_t stream) {
    TcMaps maps;
    memset(&maps, 0, sizeof maps);
    const int64_t heads = (int64_t)p.B * p.Hkv;
    // row groups must be whole tree nodes (rows_pg = tpg * G, tpg <= 256)
    if (p.G < 1 || p.rows_pg % p.G != 0 || p.rows_pg > kMaxRows) return cudaErrorInvalidValue;
    if (!tch::encode_q(&maps.q, p.q, p.B, p.T, p.Hq, p.G, p.rows_pg / p.G)) return cudaErrorInvalidValue;
    if (!tch::encode_kv_maps(p, heads, kTile, &maps.kc, &maps.vc, &maps.ks, &maps.vs)) return cudaErrorInvalidValue;
    const int stages = tc_stages(p.B, grid);
    if (stages == 5)
        return p.kv_generic ? launch_stages<5, true>(p, maps, grid, stream)
                            : launch_stages<5, false>(p, maps, grid, stream);
    if (stages == 4)
        return p.kv_generic ? launch_stages<4, true>(p, maps, grid, stream)
                            : launch_stages<4, false>(p, maps, grid, stream);
    return cudaErrorInvalidConfiguration;
}

}  // namespace hta
