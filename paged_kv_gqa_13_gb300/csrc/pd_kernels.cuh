// The kernel variants for one element type, looked up by the host code.
#pragma once

#include <type_traits>

#include "pd_decode.cuh"
#include "pd_decode_mma.cuh"
#include "pd_merge.cuh"

namespace pd {

// Kernels and sizes for one (T, head_dim, heads per tile) combination.
struct KernelSet {
    const void* decode;
    const void* variant[4];  // decode kernel per variant bits (variant[0] == decode)
    const void* merge;
    const void* merge_states;
    int warp_bytes;      // dynamic shared memory per decode warp
    int rows_per_stage;  // K (and V) rows one pipeline stage holds
    int mma;             // 1: tensor-core kernel (K/V always through 128B-swizzled tensor maps)
    int smem_slack;      // extra dynamic shared memory for aligning the stages
};

template <typename T>
bool lookup_kernels_t(int D, int G, KernelSet* ks) {
    constexpr bool kHalf = sizeof(T) == 2;
#define PD_CASE(DD, GG)                                                                 \
    if (D == DD && G == GG) {                                                           \
        ks->merge = reinterpret_cast<const void*>(merge_partials_kernel<T, DD>);        \
        ks->merge_states = reinterpret_cast<const void*>(merge_states_kernel<T, DD>);   \
        if constexpr (kHalf && GG == 8) {                                               \
            ks->decode = reinterpret_cast<const void*>(decode_mma_kernel<T, DD, 0>);     \
            ks->warp_bytes = CfgMma<T, DD>::kWarpBytes;                                 \
            ks->rows_per_stage = kMmaRows;                                              \
            ks->mma = 1;                                                                \
            ks->smem_slack = 1024;                                                      \
        } else {                                                                        \
            ks->decode = reinterpret_cast<const void*>(decode_kernel<T, DD, GG, 0>);     \
            ks->warp_bytes = Cfg<T, DD, GG>::kWarpBytes;                                \
            ks->rows_per_stage = Cfg<T, DD, GG>::kRC;                                   \
            ks->mma = 0;                                                                \
            ks->smem_slack = 0;                                                         \
        }                                                                               \
        return true;                                                                    \
    }
    PD_CASE(64, 1) PD_CASE(64, 2) PD_CASE(64, 4) PD_CASE(64, 8)
    PD_CASE(128, 1) PD_CASE(128, 2) PD_CASE(128, 4) PD_CASE(128, 8)
    PD_CASE(256, 1) PD_CASE(256, 2) PD_CASE(256, 4) PD_CASE(256, 8)
#undef PD_CASE
    return false;
}

// The decode kernel of one variant (kVarFused / kVarNhd bits, not 0) for
// (T, head_dim, heads per tile); its shared-memory layout is that of the plain
// kernel of lookup_kernels_t. Each variant is instantiated in a translation
// unit of its own, so that the variants build in parallel.
template <typename T, int kVariant>
bool lookup_variant_t(int D, int G, const void** fn) {
    constexpr bool kHalf = sizeof(T) == 2;
#define PD_CASE(DD, GG)                                                                 \
    if (D == DD && G == GG) {                                                           \
        if constexpr (kHalf && GG == 8)                                                 \
            *fn = reinterpret_cast<const void*>(decode_mma_kernel<T, DD, kVariant>);    \
        else                                                                            \
            *fn = reinterpret_cast<const void*>(decode_kernel<T, DD, GG, kVariant>);    \
        return true;                                                                    \
    }
    PD_CASE(64, 1) PD_CASE(64, 2) PD_CASE(64, 4) PD_CASE(64, 8)
    PD_CASE(128, 1) PD_CASE(128, 2) PD_CASE(128, 4) PD_CASE(128, 8)
    PD_CASE(256, 1) PD_CASE(256, 2) PD_CASE(256, 4) PD_CASE(256, 8)
#undef PD_CASE
    return false;
}

}  // namespace pd
