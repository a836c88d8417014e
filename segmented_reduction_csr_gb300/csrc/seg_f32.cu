// seg_f32.cu -- float instantiations of the segmented-reduction kernel.
#include "seg_pick.cuh"

namespace segred {
const void* pick_kernel_f32(int op, int off_is_i64, int shape) {
    return pick_kernel<float>(op, off_is_i64, shape);
}
}  // namespace segred
