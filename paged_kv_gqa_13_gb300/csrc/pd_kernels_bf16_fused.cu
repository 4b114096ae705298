// Fused append + decode kernels for element type __nv_bfloat16.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_fused_bf16(int head_dim, int heads, const void** fn) {
    return lookup_variant_t<__nv_bfloat16, 1>(head_dim, heads, fn);
}
}  // namespace pd
