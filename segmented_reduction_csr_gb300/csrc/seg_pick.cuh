// seg_pick.cuh -- maps (op, offsets type, kernel shape) to one instantiation
// of seg_reduce_kernel for a value type.  Each value type is compiled in its
// own translation unit (seg_u32.cu, seg_s32.cu, seg_f32.cu) so the builds
// run in parallel.
#pragma once
#include "seg_rows2.cuh"
#include "seg_scalar.cuh"
#include "seg_small.cuh"

namespace segred {

// Kernel shapes; the host planner picks one (seg_plan_t::kernel_variant).
enum : int {
    SHAPE_ROWS_VEC1 = 0,    // F > 1: one 32-bit column per lane, register ring
    SHAPE_ROWS_VEC2 = 1,    // F > 1, F even, 8-byte aligned rows: two columns per lane
    SHAPE_ROWS_VEC4 = 2,    // F > 1, F % 4 == 0, 16-byte aligned rows: four columns per lane
    SHAPE_SCALAR = 4,       // F == 1: the scalar kernel
    SHAPE_STAGED_VEC1 = 5,  // 1 < F <= 32, F % 4 == 0, 16-byte aligned: rows staged by bulk copies
    SHAPE_STAGED_VEC2 = 6,  // 32 < F <= 64, same
    SHAPE_STAGED_VEC4 = 7,  // 64 < F <= 128, same
    SHAPE_SMALL = 8,        // F == 1, at most SM_MAXR rows and SM_MAXS segments: one CTA
    SHAPE_COUNT = 9
};

template <class T, int OP, class OffT>
const void* pick_shape(int shape) {
    switch (shape) {
        case SHAPE_ROWS_VEC1: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 1, false>);
        case SHAPE_ROWS_VEC2: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 2, false>);
        case SHAPE_ROWS_VEC4: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 4, false>);
        case SHAPE_SCALAR: return reinterpret_cast<const void*>(&seg_scalar_kernel<T, OP, OffT>);
        case SHAPE_STAGED_VEC1: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 1, true>);
        case SHAPE_STAGED_VEC2: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 2, true>);
        case SHAPE_STAGED_VEC4: return reinterpret_cast<const void*>(&seg_rows2_kernel<T, OP, OffT, 4, true>);
        case SHAPE_SMALL: return reinterpret_cast<const void*>(&seg_small_kernel<T, OP, OffT>);
        default: return nullptr;
    }
}

template <class T, class OffT>
const void* pick_op(int op, int shape) {
    switch (op) {
        case OP_SUM: return pick_shape<T, OP_SUM, OffT>(shape);
        case OP_MIN: return pick_shape<T, OP_MIN, OffT>(shape);
        case OP_MAX: return pick_shape<T, OP_MAX, OffT>(shape);
        default: return nullptr;
    }
}

template <class T>
const void* pick_kernel(int op, int off_is_i64, int shape) {
    return off_is_i64 ? pick_op<T, int64_t>(op, shape) : pick_op<T, uint32_t>(op, shape);
}

// Defined in seg_u32.cu / seg_s32.cu / seg_f32.cu.
const void* pick_kernel_u32(int op, int off_is_i64, int shape);
const void* pick_kernel_s32(int op, int off_is_i64, int shape);
const void* pick_kernel_f32(int op, int off_is_i64, int shape);

}  // namespace segred
