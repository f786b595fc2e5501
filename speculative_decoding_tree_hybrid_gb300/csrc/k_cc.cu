// CUDA-core (FFMA) path of the hybrid tree attention, for head dimension 64
// and for trees whose packed query rows are too few to fill a tensor-core
// tile. One persistent cooperative grid covers both parts of the method
// ("LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", Korean summary section 2.C: the unmasked cached
// part and the masked speculative part) as tiles of 64 keys, then merges all
// partial softmaxes with the log-sum-exp rule after a grid barrier.
//
// Block: 8 warps; a row group holds up to 32 packed query rows, 4 per warp.
// Per 64-key tile: K and V are staged in shared memory (K rows padded so
// 16-byte reads of 8 consecutive rows hit distinct banks), each lane scores
// keys lane and lane+32 against its warp's 4 rows, the warp keeps an online
// softmax in base 2 (scores pre-multiplied by scale*log2 e), and each lane
// accumulates d/32 adjacent output columns.
#include "hta_internal.cuh"
#include "hta_launch.h"

namespace hta {
namespace {

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

// Processes units [u_begin, u_end) of one segment with the CTA's 32-row group.
template <int D>
__device__ __forceinline__ void cc_piece(const AttnParams &p, CcSmem<D> &sm, int32_t b, int32_t kvh, int32_t rg,
                         int32_t Lb, int32_t u_begin, int32_t u_end, RowState<D> &st) {
    constexpr int CPL = D / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrows = rows_in_group(p, rg);
    const int r_base = rg * p.rows_pg;

    // queries of this row group, scaled, zero for padding rows
    __syncthreads();
    for (int i = tid; i < kRowsPerGroup * (D / 8); i += kThreads) {
        const int lr = i / (D / 8), c8 = (i % (D / 8)) * 8;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (lr < nrows) {
            const int r = r_base + lr, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
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
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        st.m[i] = -INFINITY;
        st.l[i] = 0.f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) st.acc[i][k] = 0.f;
    }

    const int n_tree = p.include_tree ? p.n_tree_tiles : 0;
    const int64_t kv_off = ((int64_t)b * p.Hkv + kvh);
    for (int u = u_begin; u < u_end; ++u) {
        const bool tree = u < n_tree;
        const int j0 = (tree ? u : u - n_tree) * kTile;
        const int nvalid = tree ? min(kTile, p.T - j0) : min(kTile, Lb - j0);
        const __nv_bfloat16 *kg = tree ? p.k_spec + (kv_off * p.T + j0) * D
                                       : p.k_cache + (kv_off * p.Lmax + j0) * D;
        const __nv_bfloat16 *vg = tree ? p.v_spec + (kv_off * p.T + j0) * D
                                       : p.v_cache + (kv_off * p.Lmax + j0) * D;
        __syncthreads();  // previous tile fully consumed
        for (int i = tid; i < kTile * (D / 8); i += kThreads) {
            const int j = i / (D / 8), c8 = (i % (D / 8)) * 8;
            uint4 kr = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
            if (j < nvalid) {
                kr = __ldg(reinterpret_cast<const uint4 *>(kg + (int64_t)j * D + c8));
                vr = __ldg(reinterpret_cast<const uint4 *>(vg + (int64_t)j * D + c8));
            }
            *reinterpret_cast<uint4 *>(&sm.k[j][c8]) = kr;
            *reinterpret_cast<uint4 *>(&sm.v[j][c8]) = vr;
        }
        __syncthreads();

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
            if (jj >= nvalid) {
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) s[i][h] = -INFINITY;
            } else if (tree) {
                const int j = j0 + jj;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const int lr = warp * kRowsPerWarp + i;
                    bool vis = false;
                    if (lr < nrows) {
                        const int t = (r_base + lr) / p.G;
                        const uint32_t w = p.mask[((int64_t)b * p.T + t) * p.W + (j >> 5)];
                        vis = (w >> (j & 31)) & 1u;
                    }
                    if (!vis) s[i][h] = -INFINITY;
                }
            }
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
}

// Writes the row state of a finished piece: a partial (split mode) or the
// normalised output (direct mode, the CTA saw every unit of the segment).
template <int D>
__device__ __forceinline__ void cc_emit(const AttnParams &p, const RowState<D> &st, int64_t seg, int32_t b,
                        int32_t kvh, int32_t rg, int64_t slot, bool direct) {
    constexpr int CPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = rows_in_group(p, rg);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int lr = warp * kRowsPerWarp + i;
        if (lr >= nrows) continue;
        if (!direct) {
            float *rec = p.ws_rec + (slot * p.rows_pg + lr) * (D + 4);
#pragma unroll
            for (int k = 0; k < CPL; ++k) rec[lane * CPL + k] = st.acc[i][k];
            if (lane == 0) {
                rec[D] = st.m[i];
                rec[D + 1] = st.l[i];
            }
        } else {
            const int r = rg * p.rows_pg + lr, t = r / p.G, hq = kvh * p.G + (r - t * p.G);
            const int64_t out_row = ((int64_t)b * p.T + t) * p.Hq + hq;
            const bool any = st.l[i] > 0.f;
            const float inv = any ? 1.f / st.l[i] : 0.f;
            const float lse = any ? (st.m[i] + log2f(st.l[i])) * kLn2 : -INFINITY;
            if (p.out_fp32) {
                float *o = (float *)p.out_o + out_row * D + lane * CPL;
#pragma unroll
                for (int k = 0; k < CPL; ++k) o[k] = st.acc[i][k] * inv;
            } else {
                __nv_bfloat16 *o = (__nv_bfloat16 *)p.out_o + out_row * D + lane * CPL;
#pragma unroll
                for (int k = 0; k < CPL; k += 2)
                    *reinterpret_cast<__nv_bfloat162 *>(o + k) =
                        __floats2bfloat162_rn(st.acc[i][k] * inv, st.acc[i][k + 1] * inv);
            }
            if (lane == 0) p.out_lse[out_row] = lse;
        }
    }
    (void)seg;
}

template <int D>
__global__ void __launch_bounds__(kThreads) k_cc_attn(const __grid_constant__ AttnParams p, int direct) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    CcSmem<D> &sm = *reinterpret_cast<CcSmem<D> *>(smem_raw);
    RowState<D> st;

    if (direct) {
        // every CTA owns whole segments; no workspace, no barrier
        const int64_t n_seg = (int64_t)p.B * p.Hkv * p.n_rg;
        for (int64_t seg = blockIdx.x; seg < n_seg; seg += gridDim.x) {
            const int32_t rg = (int32_t)(seg % p.n_rg);
            const int32_t kvh = (int32_t)((seg / p.n_rg) % p.Hkv);
            const int32_t b = (int32_t)(seg / ((int64_t)p.n_rg * p.Hkv));
            int32_t Lb = 0;
            if (p.include_cache) {
                Lb = p.cache_lens[b];
                if (Lb < 0 || (int64_t)Lb > p.Lmax) {
                    if (kvh == 0 && rg == 0 && threadIdx.x == 0) flag_error(p.dev_err, HTA_DEVERR_CACHE_LEN);
                    Lb = Lb < 0 ? 0 : (int32_t)p.Lmax;
                }
            }
            cc_piece<D>(p, sm, b, kvh, rg, Lb, 0, seg_units(p, Lb), st);
            cc_emit<D>(p, st, seg, b, kvh, rg, 0, true);
        }
        return;
    }

    int32_t *lens_s = reinterpret_cast<int32_t *>(smem_raw + sizeof(CcSmem<D>));
    int64_t *pre_s = reinterpret_cast<int64_t *>(smem_raw + sizeof(CcSmem<D>) +
                                                 ((p.B * 4 + 15) / 16) * 16);
    int64_t *lo_s = pre_s + p.B + 1;
    build_schedule(p, lens_s, pre_s, lo_s);
    int64_t u = lo_s[blockIdx.x];
    const int64_t u_end = lo_s[blockIdx.x + 1];
    while (u < u_end) {
        const UnitPos pos = locate_unit(p, u, lens_s, pre_s);
        const int64_t seg_end = pos.seg_begin + pos.seg_units;
        const int64_t piece_end = seg_end < u_end ? seg_end : u_end;
        const int32_t n = (int32_t)(piece_end - u);
        cc_piece<D>(p, sm, pos.b, pos.kvh, pos.rg, lens_s[pos.b], pos.unit, pos.unit + n, st);
        cc_emit<D>(p, st, pos.seg, pos.b, pos.kvh, pos.rg, slot_of(p, pos.seg, blockIdx.x), false);
        u = piece_end;
    }
    __syncthreads();  // the tile buffers stage the merge
    static_assert(sizeof(CcSmem<D>) >= kMergePlanBytes + 32 * (D + 4) * 4, "merge stage too small");
    merge_phase<D>(p, lens_s, pre_s, lo_s, smem_raw, (uint32_t)sizeof(CcSmem<D>));
    grid_barrier_depart(p);
}

template <int D>
size_t cc_smem_bytes(int B, int grid) {
    return sizeof(CcSmem<D>) + sched_bytes(B, grid);
}

template <int D>
cudaError_t cc_launch_t(const AttnParams &p, bool direct, int grid, cudaStream_t stream) {
    const size_t smem = cc_smem_bytes<D>(p.B, grid);
    cudaError_t e = cudaFuncSetAttribute(k_cc_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = direct ? 0 : 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_cc_attn<D>, p, direct ? 1 : 0);
}

template <int D>
int cc_max_grid_t(int B, int num_sms) {
    // the boundary table grows with the grid: size it for 8 CTAs per SM
    const size_t smem = cc_smem_bytes<D>(B, 8 * num_sms);
    if (cudaFuncSetAttribute(k_cc_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_cc_attn<D>, kThreads, smem) != cudaSuccess)
        return 0;
    return (occ < 8 ? occ : 8) * num_sms;
}

}  // namespace

int cc_rows_per_group() { return kRowsPerGroup; }
int cc_tile() { return kTile; }

int cc_max_grid(int d, int B, int num_sms) {
    return d == 128 ? cc_max_grid_t<128>(B, num_sms) : cc_max_grid_t<64>(B, num_sms);
}

cudaError_t cc_launch(const AttnParams &p, bool direct, int grid, cudaStream_t stream) {
    return p.d == 128 ? cc_launch_t<128>(p, direct, grid, stream) : cc_launch_t<64>(p, direct, grid, stream);
}

}  // namespace hta
