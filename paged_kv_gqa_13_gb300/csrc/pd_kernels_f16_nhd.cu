// NHD contiguous decode kernels for element type __half.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_nhd_f16(int head_dim, int heads, const void** fn) {
    return lookup_variant_t<__half, 2>(head_dim, heads, fn);
}
}  // namespace pd
