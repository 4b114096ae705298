// NHD contiguous decode kernels for element type float.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_nhd_f32(int head_dim, int heads, const void** fn) {
    return lookup_variant_t<float, 2>(head_dim, heads, fn);
}
}  // namespace pd
