// C-ABI entry points of libhta: argument checks, workspace layout, kernel-path
// choice and launches. Every step of the computation runs in the kernels of
// k_mask.cu, k_cc.cu, k_tc.cu, k_tc2.cu, k_merge.cu, k_accept.cu, k_window.cu and k_lspec.cu; this file only validates and
// dispatches.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <initializer_list>

#include "hta_launch.h"

using hta::AttnParams;

namespace {

thread_local int32_t g_last_path = 0;

constexpr size_t kWsAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// int32 / fp32 arrays (NULL entries are optional arguments and pass)
bool aligned4(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (((uintptr_t)p & 3u) != 0) return false;
    return true;
}

// Memory of the current device (NULL passes: optional arguments). The
// tensor-core kernels read their inputs through TMA tensor maps, and the
// clustered one multicasts each tile to the CTAs of a cluster; those maps
// must cover this GPU's own memory only.
bool on_current_device(std::initializer_list<const void *> ps) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    for (const void *ptr : ps) {
        if (!ptr) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != dev) return false;
    }
    return true;
}

int num_sms_current() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

bool tc_device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3;
}

hta_status check_dims(const hta_dims *d) {
    if (!d) return HTA_ERR_INVALID_ARG;
    if (d->B <= 0 || d->T <= 0 || d->Hq <= 0 || d->Hkv <= 0 || d->d <= 0 || d->Lmax < 0)
        return HTA_ERR_INVALID_ARG;
    if (!(d->scale >= 0.f) || isinf(d->scale)) return HTA_ERR_INVALID_ARG;
    if (d->Hq % d->Hkv != 0) return HTA_ERR_UNSUPPORTED;
    if (d->d != 64 && d->d != 128) return HTA_ERR_UNSUPPORTED;
    if (d->T > HTA_TMAX || d->B > HTA_BMAX) return HTA_ERR_UNSUPPORTED;
    if (d->Lmax > (int64_t)0x7fffffff) return HTA_ERR_UNSUPPORTED;
    return HTA_OK;
}

// The storage rules of hta_kv_layout; NULL = contiguous head-major.
hta_status check_layout(const hta_dims *d, const hta_kv_layout *l) {
    if (!l) return HTA_OK;
    if (l->order != HTA_KV_HND && l->order != HTA_KV_NHD) return HTA_ERR_INVALID_ARG;
    if (l->page_size < 0) return HTA_ERR_INVALID_ARG;
    if (l->page_size == 0) return HTA_OK;
    const int32_t P = l->page_size;
    // a 128-key tile covers whole pages, or lies inside one
    if (!(P == 16 || P == 32 || P == 64 || P % 128 == 0)) return HTA_ERR_INVALID_ARG;
    if (!l->block_table || l->max_pages <= 0 || l->num_pages <= 0) return HTA_ERR_INVALID_ARG;
    if (!aligned4({l->block_table})) return HTA_ERR_ALIGN;
    if (d->Lmax > (int64_t)l->max_pages * P) return HTA_ERR_INVALID_ARG;
    return HTA_OK;
}

void apply_layout(AttnParams &p, const hta_kv_layout *l) {
    if (!l) return;
    p.kv_nhd = l->order == HTA_KV_NHD ? 1 : 0;
    p.page_size = l->page_size;
    if (l->page_size > 0) {
        p.max_pages = l->max_pages;
        p.num_pages = l->num_pages;
        p.block_table = l->block_table;
    }
    p.kv_generic = (p.kv_nhd || p.page_size > 0) ? 1 : 0;
}

enum Path { kPathNone = 0, kPathCC = 1, kPathTC = 2, kPathTC2 = 3 };

// Environment override HTA_FORCE_PATH=cc|tc|tc2, read on every call.
int forced_path() {
    const char *s = getenv("HTA_FORCE_PATH");
    if (!s) return kPathNone;
    if (!strcmp(s, "cc")) return kPathCC;
    if (!strcmp(s, "tc")) return kPathTC;
    if (!strcmp(s, "tc2")) return kPathTC2;
    return kPathNone;
}

// Tensor cores whenever the head dimension is 128: even a decode-shaped call
// (a few packed rows per KV head) streams the cache faster through the TMA
// pipeline of the tensor-core kernel (its 128-row tile has room to spare) than
// through the CUDA-core kernel. Past 128 rows, pairs of SMs that share every
// K/V tile (one 128-row sub-group each, 2 to 4 per cluster), when such
// clusters fit on the device.
// CTAs per cluster of the clustered kernel: enough 128-row sub-groups (whole
// tree nodes each) to hold every packed row of a KV head, 2 to 4; a larger
// tree is split into row groups that each stream the cache
int tc2_csize(const hta_dims *d) {
    const int G = d->Hq / d->Hkv, nodes = hta::tc2_rows_per_sub() / G;  // tree nodes per CTA
    if (nodes < 1) return 2;
    const int need = (d->T + nodes - 1) / nodes;
    return need < 2 ? 2 : need > 4 ? 4 : need;
}

bool tc2_fits(const hta_dims *d) {
    const int G = d->Hq / d->Hkv, c = tc2_csize(d);
    return G <= 64 && hta::tc2_max_grid(d->B, num_sms_current(), c) >= c;
}

int choose_path(const hta_dims *d) {
    const int forced = forced_path();
    const int G = d->Hq / d->Hkv, R = d->T * G;
    const bool tc_ok = d->d == 128 && tc_device_ok() && hta::tc_rows_per_group() > 0;
    if (forced == kPathCC) return kPathCC;
    if (forced == kPathTC) return (tc_ok && G <= hta::tc_rows_per_group()) ? kPathTC : kPathNone;
    if (forced == kPathTC2) return (tc_ok && R > 128 && tc2_fits(d)) ? kPathTC2 : kPathNone;
    if (tc_ok && R > 128 && tc2_fits(d)) return kPathTC2;
    return (tc_ok && G <= hta::tc_rows_per_group()) ? kPathTC : kPathCC;
}

struct Layout {
    int n_rg, rows_pg, tile, n_tree_tiles, subs;
    int64_t n_seg, slots;
    size_t off_rec, total;
};

Layout make_layout(const hta_dims *d, int path, int grid, bool tree) {
    Layout L = {};
    const int R = d->T * (d->Hq / d->Hkv);
    const int rpg_max = path == kPathTC ? hta::tc_rows_per_group() : hta::cc_rows_per_group();
    L.tile = path == kPathTC ? hta::tc_tile() : path == kPathTC2 ? hta::tc2_tile() : hta::cc_tile();
    if (path == kPathTC2) {
        // whole tree nodes per group, each half of a group at most one
        // 128-row MMA tile
        const int G = d->Hq / d->Hkv, tpg_max = tc2_csize(d) * (hta::tc2_rows_per_sub() / G);
        L.n_rg = (d->T + tpg_max - 1) / tpg_max;
        L.rows_pg = (d->T + L.n_rg - 1) / L.n_rg * G;
    } else if (path == kPathTC) {
        // whole tree nodes per group: the tensor-core path loads a group's Q
        // rows as one box of tpg nodes x G heads
        const int G = d->Hq / d->Hkv, tpg_max = rpg_max / G;
        L.n_rg = (d->T + tpg_max - 1) / tpg_max;
        L.rows_pg = (d->T + L.n_rg - 1) / L.n_rg * G;
    } else {
        L.n_rg = (R + rpg_max - 1) / rpg_max;
        L.rows_pg = (R + L.n_rg - 1) / L.n_rg;
    }
    L.n_tree_tiles = tree ? (d->T + L.tile - 1) / L.tile : 0;
    L.n_seg = (int64_t)d->B * d->Hkv * L.n_rg;
    // record slots: (segment + worker) * records per piece, a staircase of
    // pieces (the clustered kernel has grid / csize workers)
    L.subs = 1;
    L.slots = (L.n_seg + (path == kPathTC2 ? grid / tc2_csize(d) : grid)) * L.subs;
    // [barrier counters | partial records (d + 4 floats per row)]
    L.off_rec = kWsAlign;
    L.total = align_up(L.off_rec + (size_t)L.slots * L.rows_pg * (d->d + 4) * sizeof(float), kWsAlign);
    return L;
}

int max_grid(int path, const hta_dims *d) {
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    if (path == kPathTC2) return hta::tc2_max_grid(d->B, sms, tc2_csize(d));
    return path == kPathTC ? hta::tc_max_grid(d->B, sms) : hta::cc_max_grid(d->d, d->B, sms);
}

// Bound of the grid-barrier wait before the merge: ~4 s of SM cycles, or
// HTA_TEST_BARRIER_WAIT_CYCLES (read on every call) for failure-detection
// tests that make that wait run out on purpose.
uint64_t barrier_wait_cycles() {
    const char *s = getenv("HTA_TEST_BARRIER_WAIT_CYCLES");
    if (s && *s) {
        char *end = nullptr;
        const unsigned long long v = strtoull(s, &end, 10);
        if (end && *end == 0) return (uint64_t)v;
    }
    return 8000000000ull;
}

// The largest grid no larger than `grid` (whole clusters on the clustered
// path) whose workspace layout fits in ws_bytes; 0 when not even one worker
// fits.
int fit_grid(const hta_dims *d, int path, int grid, bool tree, size_t ws_bytes) {
    const Layout L0 = make_layout(d, path, 0, tree);
    const size_t per_slot = (size_t)L0.rows_pg * (d->d + 4) * sizeof(float);
    const size_t usable = ws_bytes / kWsAlign * kWsAlign;
    if (usable <= L0.off_rec || per_slot == 0) return 0;
    const int64_t slots = (int64_t)((usable - L0.off_rec) / per_slot);
    const int64_t workers = slots / (L0.subs > 0 ? L0.subs : 1) - L0.n_seg;
    if (workers < 1) return 0;
    const int c = path == kPathTC2 ? tc2_csize(d) : 1;
    const int64_t w = workers < (int64_t)(grid / c) ? workers : grid / c;
    return (int)(w * c);
}

AttnParams base_params(const hta_dims *d, const Layout &L) {
    AttnParams p;
    memset(&p, 0, sizeof p);
    p.B = d->B;
    p.T = d->T;
    p.Hq = d->Hq;
    p.Hkv = d->Hkv;
    p.G = d->Hq / d->Hkv;
    p.d = d->d;
    p.W = (d->T + 31) / 32;
    p.Lmax = d->Lmax;
    const double scale = d->scale > 0.f ? (double)d->scale : 1.0 / sqrt((double)d->d);
    p.scale_log2 = (float)(scale * 1.4426950408889634);
    p.R = d->T * p.G;
    p.n_rg = L.n_rg;
    p.rows_pg = L.rows_pg;
    p.tile = L.tile;
    p.n_tree_tiles = L.n_tree_tiles;
    p.subs = L.subs > 0 ? L.subs : 1;
    p.bar_wait_cycles = barrier_wait_cycles();
    return p;
}

// Runs one attention launch over the cache and/or the tree.
hta_status run_attention(const hta_dims *d, const void *q, const void *kc, const void *vc,
                         const int32_t *lens, const void *ks, const void *vs, const uint32_t *mask,
                         void *out_o, float *out_lse, bool out_fp32, bool use_cache, bool use_tree,
                         void *ws, size_t ws_bytes, int32_t *dev_err, cudaStream_t stream,
                         const hta_kv_layout *kvl = nullptr) {
    if (!on_current_device({q, kc, vc, ks, vs})) return HTA_ERR_INVALID_ARG;
    const int path = choose_path(d);
    if (path == kPathNone) return HTA_ERR_UNSUPPORTED;
    const int gmax = max_grid(path, d);
    if (gmax <= 0) return HTA_ERR_CUDA;
    const bool direct = !use_cache;  // tree-only: one CTA finishes each segment, no workspace
    Layout L0 = make_layout(d, path, 0, use_tree);
    const int64_t max_units =
        L0.n_seg * (int64_t)(L0.n_tree_tiles + (use_cache ? (d->Lmax + L0.tile - 1) / L0.tile : 0));
    // the kernels index units and output rows with 32-bit arithmetic
    if (max_units > (int64_t)0x7fffffff || L0.n_seg * (int64_t)L0.rows_pg > (int64_t)0x7fffffff)
        return HTA_ERR_UNSUPPORTED;
    int grid;
    if (path == kPathTC2 && direct) return HTA_ERR_UNSUPPORTED;  // tree-only calls take the CUDA-core path
    if (direct)
        grid = (int)(L0.n_seg < (int64_t)gmax ? L0.n_seg : gmax);
    else if (path == kPathTC2) {  // one worker per cluster
        const int c = tc2_csize(d);
        grid = c * (int)(max_units < (int64_t)(gmax / c) ? (max_units > 0 ? max_units : 1) : gmax / c);
    }
    else
        grid = (int)(max_units < (int64_t)gmax ? (max_units > 0 ? max_units : 1) : gmax);
    if (!direct && ws && ((uintptr_t)ws % kWsAlign) == 0) {
        // A workspace sized for shorter lengths than Lmax holds fewer record
        // slots: run with the workers it holds (fewer workers only matter when
        // the lengths have more tiles than workers)
        const int fit = fit_grid(d, path, grid, use_tree, ws_bytes);
        if (fit > 0 && fit < grid) grid = fit;
    }
    Layout L = make_layout(d, path, grid, use_tree);
    AttnParams p = base_params(d, L);
    p.csize = path == kPathTC2 ? tc2_csize(d) : 0;
    p.workers = path == kPathTC2 ? grid / p.csize : grid;
    p.q = (const __nv_bfloat16 *)q;
    p.k_cache = (const __nv_bfloat16 *)kc;
    p.v_cache = (const __nv_bfloat16 *)vc;
    p.cache_lens = lens;
    p.k_spec = (const __nv_bfloat16 *)ks;
    p.v_spec = (const __nv_bfloat16 *)vs;
    p.mask = mask;
    p.out_o = out_o;
    p.out_lse = out_lse;
    p.out_fp32 = out_fp32 ? 1 : 0;
    p.include_cache = use_cache ? 1 : 0;
    p.include_tree = use_tree ? 1 : 0;
    p.dev_err = dev_err;
    apply_layout(p, kvl);
    if (!direct) {
        if (!ws || ((uintptr_t)ws % kWsAlign) != 0 || ws_bytes < L.total) return HTA_ERR_WORKSPACE;
        char *base = (char *)ws;
        p.bar = (unsigned int *)base;
        p.ws_rec = (float *)(base + L.off_rec);
        p.slots = L.slots;
    }
    cudaError_t e;
    if (path == kPathTC2) {
        e = hta::tc2_launch(p, grid, stream);
    } else if (path == kPathTC) {
        if (direct) return HTA_ERR_UNSUPPORTED;  // tree-only calls take the CUDA-core path
        e = hta::tc_launch(p, grid, stream);
    } else {
        e = hta::cc_launch(p, direct, grid, stream);
    }
    if (e != cudaSuccess) return HTA_ERR_CUDA;
    g_last_path = path;
    return HTA_OK;
}

}  // namespace

extern "C" {

const char *hta_status_string(hta_status s) {
    switch (s) {
        case HTA_OK: return "ok";
        case HTA_ERR_INVALID_ARG: return "invalid argument";
        case HTA_ERR_UNSUPPORTED: return "unsupported shape or device";
        case HTA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case HTA_ERR_BAD_TREE: return "invalid parent array";
        case HTA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case HTA_ERR_CUDA: return "CUDA launch failed";
        case HTA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int32_t hta_last_path(void) { return g_last_path; }

hta_status hta_build_mask(const int32_t *parents, int32_t B, int32_t T, uint32_t *mask,
                          int32_t *dev_err, cudaStream_t stream) {
    if (!parents || !mask || B <= 0 || T <= 0) return HTA_ERR_INVALID_ARG;
    if (!aligned4({parents, mask, dev_err})) return HTA_ERR_ALIGN;
    if (T > HTA_TMAX || B > HTA_BMAX) return HTA_ERR_UNSUPPORTED;
    if (hta::mask_launch(parents, B, T, mask, dev_err, stream) != cudaSuccess) return HTA_ERR_CUDA;
    return HTA_OK;
}

hta_status hta_accept_commit(const hta_dims *d, const int32_t *parents, const int32_t *draft,
                             const int32_t *target, const hta_bf16 *k_spec, const hta_bf16 *v_spec,
                             hta_bf16 *k_cache, hta_bf16 *v_cache, int32_t *cache_lens, int32_t *accepted,
                             int32_t *n_accepted, int32_t *next_token, int32_t *dev_err,
                             cudaStream_t stream) {
    return hta_accept_commit_kv(d, nullptr, parents, draft, target, k_spec, v_spec, k_cache, v_cache, cache_lens,
                                accepted, n_accepted, next_token, dev_err, stream);
}

hta_status hta_accept_commit_kv(const hta_dims *d, const hta_kv_layout *layout, const int32_t *parents,
                                const int32_t *draft, const int32_t *target, const hta_bf16 *k_spec,
                                const hta_bf16 *v_spec, hta_bf16 *k_cache, hta_bf16 *v_cache, int32_t *cache_lens,
                                int32_t *accepted, int32_t *n_accepted, int32_t *next_token, int32_t *dev_err,
                                cudaStream_t stream) {
    if (!d || !parents || !draft || !target || !k_spec || !v_spec || !k_cache || !v_cache || !cache_lens ||
        !accepted || !n_accepted || !next_token)
        return HTA_ERR_INVALID_ARG;
    if (d->B <= 0 || d->T <= 0 || d->Hkv <= 0 || d->d <= 0 || d->Lmax < 0) return HTA_ERR_INVALID_ARG;
    if (d->d != 64 && d->d != 128) return HTA_ERR_UNSUPPORTED;
    if (d->T > HTA_TMAX || d->B > HTA_BMAX || d->Lmax > (int64_t)0x7fffffff) return HTA_ERR_UNSUPPORTED;
    const hta_status ls = check_layout(d, layout);
    if (ls != HTA_OK) return ls;
    if (!aligned16(k_spec) || !aligned16(v_spec) || !aligned16(k_cache) || !aligned16(v_cache))
        return HTA_ERR_ALIGN;
    if (!aligned4({parents, draft, target, cache_lens, accepted, n_accepted, next_token, dev_err}))
        return HTA_ERR_ALIGN;
    hta::KvStore st = {};
    if (layout) {
        st.nhd = layout->order == HTA_KV_NHD ? 1 : 0;
        st.page_size = layout->page_size;
        if (layout->page_size > 0) {
            st.max_pages = layout->max_pages;
            st.num_pages = layout->num_pages;
            st.block_table = layout->block_table;
        }
    }
    if (hta::accept_launch(parents, draft, target, d->B, d->T, d->Hkv, d->d, d->Lmax, k_spec, v_spec, k_cache,
                           v_cache, cache_lens, accepted, n_accepted, next_token, dev_err, st, stream) != cudaSuccess)
        return HTA_ERR_CUDA;
    return HTA_OK;
}

hta_status hta_window_attn(const hta_dims *d, int32_t window, const hta_bf16 *q, const hta_bf16 *k_ring,
                           const hta_bf16 *v_ring, const int32_t *pos, hta_bf16 *o, float *lse, int32_t *dev_err,
                           cudaStream_t stream) {
    const hta_status st = check_dims(d);
    if (st != HTA_OK) return st;
    if (!q || !k_ring || !v_ring || !pos || !o || !lse) return HTA_ERR_INVALID_ARG;
    if (window < 1 || d->Lmax < 1) return HTA_ERR_INVALID_ARG;  // the ring holds S = Lmax slots
    // the first query still reads window - 1 positions older than itself
    if ((int64_t)window + d->T - 1 > d->Lmax) return HTA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_ring) || !aligned16(v_ring) || !aligned16(o)) return HTA_ERR_ALIGN;
    if (!aligned4({pos, lse, dev_err})) return HTA_ERR_ALIGN;
    Layout L = {};
    L.n_rg = 1;
    L.rows_pg = d->T * (d->Hq / d->Hkv);
    AttnParams p = base_params(d, L);
    p.q = (const __nv_bfloat16 *)q;
    p.k_cache = (const __nv_bfloat16 *)k_ring;
    p.v_cache = (const __nv_bfloat16 *)v_ring;
    p.out_o = o;
    p.out_lse = lse;
    p.dev_err = dev_err;
    if (hta::window_launch(p, pos, window, (int32_t)d->Lmax, stream) != cudaSuccess) return HTA_ERR_CUDA;
    g_last_path = kPathCC;
    return HTA_OK;
}

hta_status hta_logitspec_tree(int32_t B, int32_t V, int64_t Lh_max, int32_t T, int32_t k, int32_t m,
                              const float *logits, const int32_t *hist, const int32_t *hist_len,
                              const int32_t *keep, int32_t *parents, int32_t *tokens, int32_t *n_nodes,
                              int32_t *next_token, int32_t *dev_err, cudaStream_t stream) {
    if (!logits || !hist || !hist_len || !keep || !parents || !tokens || !n_nodes || !next_token)
        return HTA_ERR_INVALID_ARG;
    if (B <= 0 || V <= 0 || T <= 0 || k < 0 || m <= 0 || Lh_max < 0) return HTA_ERR_INVALID_ARG;
    if (k > HTA_LSPEC_KMAX || k + 1 > V || m < 2 || m > HTA_LSPEC_MMAX || T > HTA_TMAX || B > HTA_BMAX ||
        Lh_max > (int64_t)0x7fffffff)
        return HTA_ERR_UNSUPPORTED;
    if (!aligned4({logits, hist, hist_len, parents, tokens, n_nodes, next_token, dev_err})) return HTA_ERR_ALIGN;
    hta::LspecParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r <= k; ++r) {
        if (keep[r] < 0) return HTA_ERR_INVALID_ARG;
        p.keep[r] = keep[r] < T ? keep[r] : T;
    }
    p.logits = logits;
    p.hist = hist;
    p.hist_len = hist_len;
    p.parents = parents;
    p.tokens = tokens;
    p.n_nodes = n_nodes;
    p.next_token = next_token;
    p.dev_err = dev_err;
    p.Lh_max = Lh_max;
    p.B = B;
    p.V = V;
    p.T = T;
    p.k = k;
    p.m = m;
    if (hta::lspec_launch(p, stream) != cudaSuccess) return HTA_ERR_CUDA;
    return HTA_OK;
}

size_t hta_verify_workspace_bytes(const hta_dims *d, const int32_t *host_cache_lens) {
    if (check_dims(d) != HTA_OK) return 0;
    size_t best = 0;
    const int paths[3] = {kPathCC, kPathTC, kPathTC2};
    const bool tc_ok = d->d == 128 && tc_device_ok() && hta::tc_rows_per_group() > 0;
    for (int i = 0; i < 3; ++i) {
        if (paths[i] == kPathTC && !tc_ok) continue;
        if (paths[i] == kPathTC2 && !(tc_ok && tc2_fits(d))) continue;
        int g = max_grid(paths[i], d);
        if (g <= 0) continue;
        if (host_cache_lens) {
            // a grid no larger than the units these lengths make (as the call does)
            const Layout L0 = make_layout(d, paths[i], 0, true);
            int64_t tiles = 0;
            for (int b = 0; b < d->B; ++b) {
                int64_t L = host_cache_lens[b];
                L = L < 0 ? 0 : (L > d->Lmax ? d->Lmax : L);
                tiles += L0.n_tree_tiles + (L + L0.tile - 1) / L0.tile;
            }
            const int64_t units = tiles * d->Hkv * L0.n_rg;
            if (paths[i] == kPathTC2) {
                const int c = tc2_csize(d);
                const int64_t w = units < (int64_t)(g / c) ? (units > 0 ? units : 1) : g / c;
                g = (int)(w * c);
            } else if (units < (int64_t)g) {
                g = (int)(units > 0 ? units : 1);
            }
        }
        const Layout L = make_layout(d, paths[i], g, true);
        if (L.total > best) best = L.total;
    }
    return best;
}

size_t hta_workspace_bytes(const hta_dims *d) { return hta_verify_workspace_bytes(d, nullptr); }

hta_status hta_prefix_attn(const hta_dims *d, const hta_bf16 *q, const hta_bf16 *k_cache,
                           const hta_bf16 *v_cache, const int32_t *cache_lens, float *o_c,
                           float *lse_c, void *workspace, size_t workspace_bytes,
                           int32_t *dev_err, cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if (!q || !k_cache || !v_cache || !cache_lens || !o_c || !lse_c) return HTA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_c)) return HTA_ERR_ALIGN;
    if (!aligned4({cache_lens, lse_c, dev_err})) return HTA_ERR_ALIGN;
    return run_attention(d, q, k_cache, v_cache, cache_lens, nullptr, nullptr, nullptr, o_c, lse_c,
                         true, true, false, workspace, workspace_bytes, dev_err, stream);
}

hta_status hta_tree_attn(const hta_dims *d, const hta_bf16 *q, const hta_bf16 *k_spec,
                         const hta_bf16 *v_spec, const uint32_t *mask, float *o_s, float *lse_s,
                         cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if (!q || !k_spec || !v_spec || !mask || !o_s || !lse_s) return HTA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_spec) || !aligned16(v_spec) || !aligned16(o_s)) return HTA_ERR_ALIGN;
    if (!aligned4({mask, lse_s})) return HTA_ERR_ALIGN;
    if (!on_current_device({q, k_spec, v_spec})) return HTA_ERR_INVALID_ARG;
    // the tree pass is a few MFLOP per head: it always takes the CUDA-core kernel
    hta_dims dd = *d;
    const int gmax = max_grid(kPathCC, &dd);
    if (gmax <= 0) return HTA_ERR_CUDA;
    Layout L = make_layout(&dd, kPathCC, 0, true);
    AttnParams p = base_params(&dd, L);
    p.q = (const __nv_bfloat16 *)q;
    p.k_spec = (const __nv_bfloat16 *)k_spec;
    p.v_spec = (const __nv_bfloat16 *)v_spec;
    p.mask = mask;
    p.out_o = o_s;
    p.out_lse = lse_s;
    p.out_fp32 = 1;
    p.include_cache = 0;
    p.include_tree = 1;
    const int grid = (int)(L.n_seg < (int64_t)gmax ? L.n_seg : gmax);
    if (hta::cc_launch(p, true, grid, stream) != cudaSuccess) return HTA_ERR_CUDA;
    g_last_path = kPathCC;
    return HTA_OK;
}

hta_status hta_merge(const hta_dims *d, const float *o_c, const float *lse_c, const float *o_s,
                     const float *lse_s, hta_bf16 *o, float *lse, cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if (!o_c || !lse_c || !o_s || !lse_s || !o || !lse) return HTA_ERR_INVALID_ARG;
    if (!aligned16(o_c) || !aligned16(o_s) || !aligned16(o)) return HTA_ERR_ALIGN;
    if (!aligned4({lse_c, lse_s, lse})) return HTA_ERR_ALIGN;
    const int64_t rows = (int64_t)d->B * d->T * d->Hq;
    if (hta::merge2_launch(rows, d->d, o_c, lse_c, o_s, lse_s, (__nv_bfloat16 *)o, lse, stream) !=
        cudaSuccess)
        return HTA_ERR_CUDA;
    return HTA_OK;
}

hta_status hta_verify(const hta_dims *d, const hta_bf16 *q, const hta_bf16 *k_cache,
                      const hta_bf16 *v_cache, const int32_t *cache_lens, const hta_bf16 *k_spec,
                      const hta_bf16 *v_spec, const uint32_t *mask, hta_bf16 *o, float *lse,
                      void *workspace, size_t workspace_bytes, int32_t *dev_err,
                      cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if (!q || !k_cache || !v_cache || !cache_lens || !k_spec || !v_spec || !mask || !o || !lse)
        return HTA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_spec) ||
        !aligned16(v_spec) || !aligned16(o))
        return HTA_ERR_ALIGN;
    if (!aligned4({cache_lens, mask, lse, dev_err})) return HTA_ERR_ALIGN;
    return run_attention(d, q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask, o, lse, false,
                         true, true, workspace, workspace_bytes, dev_err, stream);
}

hta_status hta_verify_kv(const hta_dims *d, const hta_kv_layout *layout, const hta_bf16 *q,
                         const hta_bf16 *k_cache, const hta_bf16 *v_cache, const int32_t *cache_lens,
                         const hta_bf16 *k_spec, const hta_bf16 *v_spec, const uint32_t *mask, hta_bf16 *o,
                         float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_err,
                         cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if ((s = check_layout(d, layout)) != HTA_OK) return s;
    if (!q || !k_cache || !v_cache || !cache_lens || !k_spec || !v_spec || !mask || !o || !lse)
        return HTA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_spec) ||
        !aligned16(v_spec) || !aligned16(o))
        return HTA_ERR_ALIGN;
    if (!aligned4({cache_lens, mask, lse, dev_err})) return HTA_ERR_ALIGN;
    return run_attention(d, q, k_cache, v_cache, cache_lens, k_spec, v_spec, mask, o, lse, false,
                         true, true, workspace, workspace_bytes, dev_err, stream, layout);
}

hta_status hta_prefix_attn_kv(const hta_dims *d, const hta_kv_layout *layout, const hta_bf16 *q,
                              const hta_bf16 *k_cache, const hta_bf16 *v_cache, const int32_t *cache_lens,
                              float *o_c, float *lse_c, void *workspace, size_t workspace_bytes,
                              int32_t *dev_err, cudaStream_t stream) {
    hta_status s = check_dims(d);
    if (s != HTA_OK) return s;
    if ((s = check_layout(d, layout)) != HTA_OK) return s;
    if (!q || !k_cache || !v_cache || !cache_lens || !o_c || !lse_c) return HTA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_c)) return HTA_ERR_ALIGN;
    if (!aligned4({cache_lens, lse_c, dev_err})) return HTA_ERR_ALIGN;
    return run_attention(d, q, k_cache, v_cache, cache_lens, nullptr, nullptr, nullptr, o_c, lse_c,
                         true, true, false, workspace, workspace_bytes, dev_err, stream, layout);
}

}  // extern "C"
