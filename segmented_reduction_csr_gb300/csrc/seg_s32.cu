// seg_s32.cu -- int32_t instantiations of the segmented-reduction kernel.
#include "seg_pick.cuh"

namespace segred {
const void* pick_kernel_s32(int op, int off_is_i64, int shape) {
    return pick_kernel<int32_t>(op, off_is_i64, shape);
}
}  // namespace segred
