// NHD contiguous fused append + decode kernels for element type float.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_nhd_fused_f32(int head_dim, int heads, const void** fn) {
    return lookup_variant_t<float, 3>(head_dim, heads, fn);
}
}  // namespace pd
