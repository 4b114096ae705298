// Decode kernels for E4M3 K/V pools with q / o of type __half.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_fp8_f16(int head_dim, int heads, bool kv_pairs, KernelSet* ks) {
    return lookup_fp8_t<__half>(head_dim, heads, kv_pairs, ks);
}
}  // namespace pd
