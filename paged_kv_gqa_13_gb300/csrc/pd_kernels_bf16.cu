// Decode, merge and merge-states kernels for element type __nv_bfloat16.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_kernels_bf16(int head_dim, int heads, KernelSet* ks) {
    return lookup_kernels_t<__nv_bfloat16>(head_dim, heads, ks);
}
}  // namespace pd
