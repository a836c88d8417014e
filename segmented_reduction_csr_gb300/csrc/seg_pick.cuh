// seg_pick.cuh -- maps (op, offsets type, kernel shape) to one instantiation
// of seg_reduce_kernel for a value type.  Each value type is compiled in its
// own translation unit (seg_u32.cu, seg_s32.cu, seg_f32.cu) so the builds
// run in parallel.
#pragma once
#include "seg_rows.cuh"
#include "seg_scalar.cuh"

namespace segred {

// Kernel shapes; the host planner picks one (seg_reduce_plan_t::kernel_variant).
enum : int {
    SHAPE_VEC1_NV1 = 0,  // F == 1, or F <= 256 without 16-byte rows
    SHAPE_VEC1_NV8 = 1,  // F <= 2048 without 16-byte rows
    SHAPE_VEC4_NV1 = 2,  // F % 4 == 0, F <= 1024, 16-byte aligned values
    SHAPE_VEC4_NV2 = 3,  // F % 4 == 0, F <= 2048, 16-byte aligned values
    SHAPE_SCALAR = 4,    // F == 1: the scalar kernel
    SHAPE_COUNT = 5
};

template <class T, int OP, class OffT>
const void* pick_shape(int shape) {
    switch (shape) {
        case SHAPE_VEC1_NV1: return reinterpret_cast<const void*>(&seg_rows_kernel<T, OP, OffT, 1, 1>);
        case SHAPE_VEC1_NV8: return reinterpret_cast<const void*>(&seg_rows_kernel<T, OP, OffT, 1, 8>);
        case SHAPE_VEC4_NV1: return reinterpret_cast<const void*>(&seg_rows_kernel<T, OP, OffT, 4, 1>);
        case SHAPE_VEC4_NV2: return reinterpret_cast<const void*>(&seg_rows_kernel<T, OP, OffT, 4, 2>);
        case SHAPE_SCALAR: return reinterpret_cast<const void*>(&seg_scalar_kernel<T, OP, OffT>);
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
