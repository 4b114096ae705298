// Decode, merge and merge-states kernels for element type __half.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_kernels_f16(int head_dim, int heads, KernelSet* ks) {
    return lookup_kernels_t<__half>(head_dim, heads, ks);
}
}  // namespace pd
