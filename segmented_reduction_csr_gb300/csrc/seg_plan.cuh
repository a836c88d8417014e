// seg_plan.cuh -- the host launch planner of the segmented reduction: from
// host-known sizes, dtype, op, the alignment of the values and the SM count
// it picks the kernel shape, the grid and the scratch a launch needs.  It
// never reads device memory.  Included once, by api.cu.
#pragma once
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "../../include/seg_reduce.h"
#include "seg_pick.cuh"

namespace {

using namespace segred;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tickets sit at the start of scratch in a region sized for the largest
// number of cross-unit partial owners any launch on the device can have (one
// CTA per SM, SW_NW units per CTA in the scalar kernel), so the partials of a
// call never overlap the ticket slots of a later call with a larger grid: a
// ticket slot only ever holds (generation << 32) | count.
int64_t ticket_region_bytes(int32_t sm_count) {
    return ceil_div(int64_t(sm_count) * SW_NW * 8, 256) * 256;
}

// Planner (host only).

seg_status_t plan_launch(seg_dtype_t dtype, int64_t F, int64_t num_values,
                         seg_offset_dtype_t offsets_dtype, int64_t S, seg_op_t op,
                         uint64_t values_addr, int32_t sm_count, seg_plan_t* pl) {
    if (!pl) return SEG_ERR_INVALID_ARGUMENT;
    if (dtype != SEG_U32 && dtype != SEG_S32 && dtype != SEG_F32) return SEG_ERR_INVALID_ARGUMENT;
    if (offsets_dtype != SEG_OFF_U32 && offsets_dtype != SEG_OFF_I64) return SEG_ERR_INVALID_ARGUMENT;
    if (op != SEG_SUM && op != SEG_MIN && op != SEG_MAX && op != SEG_MEAN) return SEG_ERR_INVALID_ARGUMENT;
    if (F < 1 || num_values < 0 || S < 0 || sm_count < 1) return SEG_ERR_INVALID_ARGUMENT;
    if (op == SEG_MEAN && dtype != SEG_F32) return SEG_ERR_UNSUPPORTED;
    if (F > SEG_MAX_FEATURES) return SEG_ERR_UNSUPPORTED;
    if (offsets_dtype == SEG_OFF_U32 && num_values > int64_t(UINT32_MAX)) return SEG_ERR_INVALID_ARGUMENT;

    std::memset(pl, 0, sizeof(*pl));
    if (F == 1 && num_values <= SM_MAXR && S <= SM_MAXS) {
        // a small input: one CTA, bound by latency (no partition, no scratch use)
        pl->grid = 1;
        pl->block = SM_NT;
        pl->slot_threads = 1;
        pl->items_per_slot = 32;
        pl->vec = 1;
        pl->vecs_per_thread = 1;
        pl->max_ends = static_cast<int32_t>(S);
        pl->kernel_variant = SHAPE_SMALL;
        pl->smem_bytes = SM_SMEM;
        pl->workspace_bytes = ticket_region_bytes(sm_count);
        return SEG_OK;
    }
    if (F == 1) {
        // the scalar kernel: SW_NW warp units per CTA, each at least two chunks of
        // rows; a segment end weighs SW_CW rows in the partition
        const int64_t witems = num_values + int64_t(SW_CW) * S;
        const int64_t per_cta = int64_t(SW_NW) * SW_TROWS * 2;
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(sm_count, ceil_div(witems, per_cta)));
        // a unit's rows are addressed with 32-bit offsets inside the unit
        if (ceil_div(witems, grid * SW_NW) + 16 >= int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;
        pl->grid = static_cast<int32_t>(grid);
        pl->block = SW_NTHREADS;
        pl->slot_threads = 1;
        pl->items_per_slot = SW_KR;
        pl->vec = 1;
        pl->vecs_per_thread = 1;
        pl->max_ends = SW_EMAXT;
        pl->kernel_variant = SHAPE_SCALAR;
        pl->smem_bytes = SW_SMEM;
        pl->workspace_bytes = ticket_region_bytes(sm_count) + 2 * grid * SW_NW * int64_t(sizeof(PartElem));
        return SEG_OK;
    }
    // the row kernel: a warp per (column slice, merge range) unit.  VEC is the
    // widest load that still gives all 32 lanes a column; narrow rows fall
    // back to one column per lane so that more rows are in flight.
    // Rows of a 16-byte multiple up to 128 columns are staged through shared
    // memory by bulk copies (one slice; VEC just covers F).
    const bool staged = F % 4 == 0 && values_addr % 16 == 0 && F <= 128;
    int32_t vec = 1;
    if (staged) vec = F > 64 ? 4 : (F > 32 ? 2 : 1);
    else if (F % 4 == 0 && values_addr % 16 == 0 && F >= 128) vec = 4;
    else if (F % 2 == 0 && values_addr % 8 == 0 && F >= 64) vec = 2;
    const int64_t nsl = ceil_div(F, int64_t(32) * vec);           // column slices
    const int64_t cw = (op == SEG_MIN || op == SEG_MAX) ? RW_CW_ARG : RW_CW_SUM;   // as the kernel, args assumed
    const int64_t witems = num_values + cw * S;
    const int64_t ranges = std::max<int64_t>(1, ceil_div(witems, RW_MIN_ITEMS));
    int64_t grid = ceil_div(ranges * nsl, RW_NW);
    grid = std::max<int64_t>(grid, ceil_div(nsl, RW_NW));           // every slice gets a unit
    grid = std::min<int64_t>(grid, std::max<int64_t>(sm_count, ceil_div(nsl, RW_NW)));
    if (grid > sm_count) return SEG_ERR_UNSUPPORTED;               // tickets: one slot per unit
    const int64_t units = grid * RW_NW;
    const int64_t nr = units / nsl;                                 // ranges per slice
    // a range's rows are addressed with 32-bit offsets inside the range
    if (ceil_div(witems, nr) + 64 >= int64_t(INT32_MAX)) return SEG_ERR_UNSUPPORTED;
    const int64_t slw = int64_t(32) * vec;
    const int64_t part_bytes = 4 + ((op == SEG_MIN || op == SEG_MAX) ? 8 : 0);

    pl->grid = static_cast<int32_t>(grid);
    pl->block = RW_NTHREADS;
    pl->slot_threads = 32;
    pl->items_per_slot = staged ? static_cast<int32_t>(RW_CB / (F * 4)) : (vec == 4 ? 16 : 32);
    pl->vec = vec;
    pl->vecs_per_thread = static_cast<int32_t>(nsl);
    pl->max_ends = 0;
    if (staged)
        pl->kernel_variant = vec == 4 ? SHAPE_STAGED_VEC4 : (vec == 2 ? SHAPE_STAGED_VEC2 : SHAPE_STAGED_VEC1);
    else
        pl->kernel_variant = vec == 4 ? SHAPE_ROWS_VEC4 : (vec == 2 ? SHAPE_ROWS_VEC2 : SHAPE_ROWS_VEC1);
    pl->smem_bytes = staged ? RW_SMEM_STAGED : RW_SMEM;
    pl->workspace_bytes = ticket_region_bytes(sm_count) + 2 * units * slw * part_bytes;
    return SEG_OK;
}

}  // namespace
