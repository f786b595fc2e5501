// Pipeline helpers shared by the tensor-core kernels: bounded mbarrier waits
// and the cursor that walks a worker's unit range tile by tile, piece by
// piece (a piece is the part of one segment inside the range).
#pragma once

#include "hta_internal.cuh"
#include "tc_ptx.cuh"

namespace hta {
namespace tcp {

using namespace tc;

__device__ __forceinline__ uint32_t bar_addr(const uint64_t &b) { return smem_u32(&b); }

// Bounded wait on an mbarrier phase; false on timeout or when another warp
// has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t *abort,
                                         int32_t *dev_err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = cycles_now();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (cycles_now() - t0 > kWaitLimitCycles) {
            *abort = 1;
            flag_error(dev_err, HTA_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *dev_err) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, dev_err));
}

// Walks a unit range tile by tile, piece by piece.
struct Cursor {
    int64_t u, u_end;
    int32_t q;      // piece counter
    int32_t left;   // tiles left in the current piece
    int32_t unit;   // next unit index inside the segment
    int32_t b, kvh, rg, Lb;
    int64_t seg;
};

struct TileInfo {
    int32_t q, unit, b, kvh, rg, Lb;
    int64_t seg;
    bool first, last;
};

__device__ __forceinline__ void cursor_init(Cursor &c, int64_t u0, int64_t u1) {
    c.u = u0;
    c.u_end = u1;
    c.q = -1;
    c.left = 0;
    c.unit = 0;
    c.b = c.kvh = c.rg = c.Lb = 0;
    c.seg = 0;
}

__device__ __forceinline__ bool cursor_next(Cursor &c, const AttnParams &p, const int32_t *lens_s,
                                            const int64_t *pre_s, TileInfo &t) {
    t.first = false;
    if (c.left == 0) {
        if (c.u >= c.u_end) return false;
        const UnitPos pos = locate_unit(p, c.u, lens_s, pre_s);
        const int64_t seg_end = pos.seg_begin + pos.seg_units;
        const int64_t piece_end = seg_end < c.u_end ? seg_end : c.u_end;
        c.left = (int32_t)(piece_end - c.u);
        c.unit = pos.unit;
        c.b = pos.b;
        c.kvh = pos.kvh;
        c.rg = pos.rg;
        c.seg = pos.seg;
        c.Lb = lens_s[pos.b];
        c.q += 1;
        c.u = piece_end;
        t.first = true;
    }
    t.q = c.q;
    t.unit = c.unit;
    t.b = c.b;
    t.kvh = c.kvh;
    t.rg = c.rg;
    t.seg = c.seg;
    t.Lb = c.Lb;
    c.unit += 1;
    c.left -= 1;
    t.last = c.left == 0;
    return true;
}

// ------------------------------------------------------------ K/V layouts

// Block-table entries of one producer warp: lane i holds entry base + i of
// sequence b and, in `next`, entry base + 32 + i. Moving on to the next 32
// entries uses `next` and loads the 32 after it, so that load has a window's
// worth of tiles to land; only a jump (a new sequence) waits for a load.
struct PageWindow {
    int32_t b = -1, base = 0, entry = 0, next = 0;
};

__device__ __forceinline__ int32_t table_entry(const AttnParams &p, int32_t b, int32_t s) {
    return s < p.max_pages ? __ldg(p.block_table + (int64_t)b * p.max_pages + s) : 0;
}

// Makes the window hold the entries of slots [slot, slot + n), n <= 32, of
// sequence b. Warp-collective (same arguments in every lane).
__device__ __forceinline__ void window_cover(const AttnParams &p, PageWindow &w, int32_t b, int32_t slot, int32_t n) {
    const int32_t lane = (int32_t)(threadIdx.x & 31);
    if (b != w.b || slot < w.base || slot + n > w.base + 64) {
        w.b = b;
        w.base = slot;
        w.entry = table_entry(p, b, slot + lane);
        w.next = table_entry(p, b, slot + 32 + lane);
    } else if (slot >= w.base + 32) {
        w.base += 32;
        w.entry = w.next;
        w.next = table_entry(p, b, w.base + 32 + lane);
    }
}

// Entry of slot s (inside the window) for this lane; every lane calls it.
__device__ __forceinline__ int32_t window_entry(const PageWindow &w, int32_t s) {
    const int32_t k = s - w.base;
    const int32_t e0 = __shfl_sync(0xffffffffu, w.entry, k & 31);
    const int32_t e1 = __shfl_sync(0xffffffffu, w.next, k & 31);
    return k < 32 ? e0 : e1;
}

// Copies of one 128-key K or V tile whose first key is y (a cache token, or
// a tree token when `tree`), for every layout but contiguous head-major,
// through 4-D tensor maps: head-major (d, rows, Hkv, outer), token-major
// (d, Hkv, rows, outer), outer = the sequence or the pool page. One box per
// 64-dim half and per page the tile spans (boxes of min(page_size, 128)
// rows, at most 16), each issued by its own lane in one warp instruction:
// lane i copies half i % 2 of the rows from (i / 2) * rows. A box past the
// sequence's last page reads page 0 (those keys are masked and their V rows
// cleared like any key past the end); an entry outside the pool is flagged
// and read as page 0.
// load4(on, shared-memory offset in the tile, c0, c1, c2, c3): every lane
// calls it; the lanes with `on` issue their box.
template <typename Load4>
__device__ __forceinline__ void kv_tile_4d(const AttnParams &p, PageWindow &w, bool tree, int32_t b, int32_t kvh,
                                           int32_t y, int32_t Lb, Load4 &&load4) {
    constexpr uint32_t kHalf = 128 * 64 * 2;  // one 64-dim half of a tile
    const int32_t lane = (int32_t)(threadIdx.x & 31), h = lane & 1;
    if (tree || p.page_size == 0) {
        const bool on = lane < 2;
        if (p.kv_nhd) load4(on, h * kHalf, h * 64, kvh, y, b);
        else load4(on, h * kHalf, h * 64, y, kvh, b);
        return;
    }
    const int32_t P = p.page_size, rows = P < 128 ? P : 128;
    const int32_t pages = 128 / rows;         // pages (or 128-row parts of one) in the tile
    const bool on = lane < 2 * pages;
    const int32_t r = on ? (lane >> 1) * rows : 0;
    const int32_t j = y + r, slot0 = y / P;
    window_cover(p, w, b, slot0, P < 128 ? pages : 1);
    int32_t pg = window_entry(w, j / P);
    if (!(on && j < Lb)) {
        pg = 0;
    } else if (pg < 0 || pg >= p.num_pages) {
        flag_error(p.dev_err, HTA_DEVERR_PAGE);
        pg = 0;
    }
    const int32_t row = j % P;
    const uint32_t off = h * kHalf + (uint32_t)r * 128;
    if (p.kv_nhd) load4(on, off, h * 64, kvh, row, pg);
    else load4(on, off, h * 64, row, kvh, pg);
}

}  // namespace tcp
}  // namespace hta
