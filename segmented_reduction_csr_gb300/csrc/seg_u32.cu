// seg_u32.cu -- uint32_t instantiations of the segmented-reduction kernel.
#include "seg_pick.cuh"

namespace segred {
const void* pick_kernel_u32(int op, int off_is_i64, int shape) {
    return pick_kernel<uint32_t>(op, off_is_i64, shape);
}
}  // namespace segred
