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

}  // namespace tcp
}  // namespace hta
