// decode_common.cuh -- pieces shared by the two decode kernels (bf16 cache and FP8 cache):
// which query row and token range a work unit covers, and the per-page bookkeeping.
#pragma once

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace dec {

struct RowGeom {
    int r, b, t, j0, j1, npages, page0;
    int slot;  // partial-output slot, or -1: this unit writes the row's final output
};

// Unit -> (query row, token range [j0, j1), partial slot). With a device-built schedule the
// unit list is the preceding kernel's output; otherwise unit = row * S + split and the range
// follows split_range.
__device__ __forceinline__ RowGeom row_geometry(const DecodeArgs& p, int unit, bool report) {
    RowGeom g;
    if (p.plan_units) {  // device-built schedule
        const int4 u = p.plan_units[unit];
        g.r = u.x;
        g.j0 = u.y;
        g.j1 = u.z;
        g.slot = u.w;
    } else {  // uniform splits: unit = row * S + split
        const int S = p.num_splits;
        g.r = unit / S;
        split_range(visible_tokens(p, g.r, report), S, unit % S, &g.j0, &g.j1);
        g.slot = S > 1 ? unit : -1;
    }
    int q_len;
    row_request(p, g.r, &g.b, &g.t, &q_len);
    g.npages = (g.j1 - g.j0 + kPage - 1) / kPage;
    g.page0 = g.j0 / kPage;
    return g;
}

// Physical block of page `pg` of request b, or -1 (reported as MLA_DEV_BAD_BLOCK_ID) if the
// block-table entry is outside the cache.
__device__ __forceinline__ int page_block(const DecodeArgs& p, int b, int pg) {
    const int32_t blk = p.block_table[(size_t)b * p.max_blocks + pg];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
        return -1;
    }
    return blk;
}

// A bounded mbarrier wait taken by a whole warp: true only if every lane's wait succeeded.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* ds) {
    bool ok = ptx::wait_bar<kCluster>(bar, parity, abort, ds);
    return __all_sync(0xffffffffu, ok);
}

// Visible rows of the unit's page `page` (0 past its last page).
__device__ __forceinline__ int valid_rows(const RowGeom& g, int page) {
    return page < g.npages ? min(kPage, g.j1 - (g.j0 + kPage * page)) : 0;
}

}  // namespace dec
}  // namespace mla
