// Decode kernels for E4M3 K/V pools with q / o of type __nv_bfloat16.
#include "pd_kernels.cuh"

namespace pd {
bool lookup_fp8_bf16(int head_dim, int heads, bool kv_pairs, KernelSet* ks) {
    return lookup_fp8_t<__nv_bfloat16>(head_dim, heads, kv_pairs, ks);
}
}  // namespace pd
