// Fused append + decode kernels for element type float.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_fused_f32(int head_dim, int heads, const void** fn) {
    return lookup_variant_t<float, 1>(head_dim, heads, fn);
}
}  // namespace pd
