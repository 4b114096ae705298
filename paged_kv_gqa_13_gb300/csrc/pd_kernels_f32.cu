// Decode, merge and merge-states kernels for element type float.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_kernels_f32(int head_dim, int heads, KernelSet* ks) {
    return lookup_kernels_t<float>(head_dim, heads, ks);
}
}  // namespace pd
