// CUDA-core (FFMA) path of the hybrid tree attention, for head dimension 64
// and for trees whose packed query rows are too few to fill a tensor-core
// tile. One persistent grid (all CTAs resident) covers both parts of the method
// ("LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", Korean summary section 2.C: the unmasked cached
// part and the masked speculative part) as tiles of 64 keys, then merges all
// partial softmaxes with the log-sum-exp rule after a grid barrier.
// The per-tile work (staging, scores, online softmax, PV) is in cc_tile.cuh.
#include "cc_tile.cuh"
#include "hta_internal.cuh"
#include "hta_launch.h"

namespace hta {
namespace {

using cct::CcSmem;
using cct::RowState;
using cct::kRowsPerGroup;
using cct::kRowsPerWarp;
using cct::kThreads;
using cct::kTile;

// Processes units [u_begin, u_end) of one segment with the CTA's 32-row group.
template <int D>
__device__ __forceinline__ void cc_piece(const AttnParams &p, CcSmem<D> &sm, int32_t b, int32_t kvh, int32_t rg,
                         int32_t Lb, int32_t u_begin, int32_t u_end, RowState<D> &st) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nrows = rows_in_group(p, rg);
    const int r_base = rg * p.rows_pg;

    // queries of this row group, scaled, zero for padding rows
    __syncthreads();
    cct::load_q<D>(p, sm, b, [&](int lr, int &t, int &hq) {
        if (lr >= nrows) return false;
        const int r = r_base + lr;
        t = r / p.G;
        hq = kvh * p.G + (r - t * p.G);
        return true;
    });
    cct::reset<D>(st);

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
            if (j < nvalid && !p.kv_generic) {
                kr = __ldg(reinterpret_cast<const uint4 *>(kg + (int64_t)j * D + c8));
                vr = __ldg(reinterpret_cast<const uint4 *>(vg + (int64_t)j * D + c8));
            } else if (j < nvalid) {  // token-major or paged storage: row by row
                const int64_t off = (tree ? spec_row_off(p, b, kvh, j0 + j) : cache_row_off(p, b, kvh, j0 + j)) + c8;
                kr = __ldg(reinterpret_cast<const uint4 *>((tree ? p.k_spec : p.k_cache) + off));
                vr = __ldg(reinterpret_cast<const uint4 *>((tree ? p.v_spec : p.v_cache) + off));
            }
            *reinterpret_cast<uint4 *>(&sm.k[j][c8]) = kr;
            *reinterpret_cast<uint4 *>(&sm.v[j][c8]) = vr;
        }
        __syncthreads();
        // cache keys are all visible; tree keys per the mask row of the query's node
        cct::tile<D>(sm, st, nvalid, [&](int i, int jj) {
            if (!tree) return true;
            const int lr = warp * kRowsPerWarp + i;
            if (lr >= nrows) return false;
            const int t = (r_base + lr) / p.G, j = j0 + jj;
            const uint32_t w = p.mask[((int64_t)b * p.T + t) * p.W + (j >> 5)];
            return ((w >> (j & 31)) & 1u) != 0;
        });
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
    __syncthreads();  // the tile buffers hold the merge's run table
    static_assert(sizeof(CcSmem<D>) >= 6 * kMergeRuns * 4, "no room for the merge's run table");
    merge_phase<D, 4>(p, lens_s, pre_s, lo_s, smem_raw);
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
    attr[0].val.cooperative = (!direct && cooperative_requested()) ? 1 : 0;
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
