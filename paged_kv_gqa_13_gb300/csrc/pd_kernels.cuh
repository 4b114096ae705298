// The kernel variants for one element type, looked up by the host code.
#pragma once

#include <type_traits>

#include "pd_decode.cuh"
#include "pd_decode_fp8.cuh"
#include "pd_decode_mma.cuh"
#include "pd_decode_tc.cuh"
#include "pd_merge.cuh"

namespace pd {

// Kernels and sizes for one (T, head_dim, heads per tile) combination.
struct KernelSet {
    const void* decode;
    const void* variant[4];  // decode kernel per variant bits (variant[0] == decode)
    const void* merge;
    const void* merge_wide;  // the merge with rounds of twice the parts, for grids of one wave at 4 blocks per SM
    const void* merge_states;
    int warp_bytes;      // dynamic shared memory per decode warp
    int rows_per_stage;  // K (and V) rows one pipeline stage holds
    int mma;             // K/V copies through 128B-swizzled tensor maps: 1 16-bit pools, 2 E4M3 pools (tensor
                         // cores), 3 E4M3 pools (tcgen05, one share per block)
    int part_heads;      // heads per partial-result slot: the group tile G, or 8 for the tensor-core kernel
    int smem_slack;      // extra dynamic shared memory for aligning the stages
    int max_warps;       // shares per block the kernel is built for (one per warp unless `threads` is set)
    int threads;         // threads per block of a kernel whose shares are groups of warps (0: a warp per share);
                         // it then runs exactly max_warps shares per block
};

// Kernels and sizes for (T, head_dim, heads per tile): 16-bit tiles of 4 to
// 8 heads on tensor cores (a 16-row chunk costs ~300 instructions there
// against ~770 on CUDA cores at 4 heads), the rest on CUDA cores.
template <typename T>
bool lookup_kernels_t(int D, int G, KernelSet* ks) {
    constexpr bool kHalf = sizeof(T) == 2;
#define PD_MMA(DD)                                                                      \
    {                                                                                   \
        ks->decode = reinterpret_cast<const void*>(decode_mma_kernel<T, DD, 0>);         \
        ks->warp_bytes = CfgMma<T, DD>::kWarpBytes;                                     \
        ks->rows_per_stage = kMmaRows;                                                  \
        ks->mma = 1;                                                                    \
        ks->part_heads = 8;                                                             \
        ks->smem_slack = 1024;                                                          \
        ks->max_warps = 8;                                                              \
        ks->threads = 0;                                                                \
    }
#define PD_CC(DD, GG)                                                                   \
    {                                                                                   \
        ks->decode = reinterpret_cast<const void*>(decode_kernel<T, DD, GG, 0>);         \
        ks->warp_bytes = Cfg<T, DD, GG>::kWarpBytes;                                    \
        ks->rows_per_stage = Cfg<T, DD, GG>::kRC;                                       \
        ks->mma = 0;                                                                    \
        ks->part_heads = GG;                                                            \
        ks->smem_slack = 0;                                                             \
        ks->max_warps = 8;                                                              \
        ks->threads = 0;                                                                \
    }
#define PD_CASE(DD, GG)                                                                 \
    if (D == DD && G == GG) {                                                           \
        ks->merge = reinterpret_cast<const void*>(merge_partials_kernel<T, DD>);        \
        ks->merge_wide = reinterpret_cast<const void*>(merge_partials_kernel<T, DD, true>); \
        ks->merge_states = reinterpret_cast<const void*>(merge_states_kernel<T, DD>);   \
        if constexpr (kHalf && GG >= 4) {                                               \
            PD_MMA(DD)                                                                  \
        } else {                                                                        \
            PD_CC(DD, GG)                                                               \
        }                                                                               \
        return true;                                                                    \
    }
    PD_CASE(64, 1) PD_CASE(64, 2) PD_CASE(64, 4) PD_CASE(64, 8)
    PD_CASE(128, 1) PD_CASE(128, 2) PD_CASE(128, 4) PD_CASE(128, 8)
    PD_CASE(256, 1) PD_CASE(256, 2) PD_CASE(256, 4) PD_CASE(256, 8)
#undef PD_CASE
#undef PD_CC
#undef PD_MMA
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
        if constexpr (kHalf && GG >= 4 && (kVariant & kVarFp8) == 0)                    \
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

// The tcgen05 E4M3 kernel for bf16 q / o (null for f16, which it does not take).
template <typename T>
const void* tc_fp8_kernel() {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return reinterpret_cast<const void*>(decode_tc_fp8_kernel<T>);
    else
        return nullptr;
}

// The decode kernel for E4M3 pools with q / o of type T (16-bit). kv_pairs
// (bf16, groups of exactly 4 q heads, an even number of kv heads): head_dim 128
// goes to the tcgen05 kernel, which takes the kv heads in pairs. Other tiles of
// 4 or more q heads at head_dim 128 / 256 go to the mma.sync tensor-core kernel
// (the CUDA cores would be issue-bound there: an E4M3 byte is a whole
// element); the rest to the CUDA-core kernel. The merge kernels are those of T (from
// lookup_kernels_t), left untouched here.
template <typename T>
bool lookup_fp8_t(int D, int G, bool kv_pairs, KernelSet* ks) {
    static_assert(sizeof(T) == 2, "E4M3 pools take 16-bit q / o");
#define PD_CASE(DD, GG)                                                                      \
    if (D == DD && G == GG) {                                                                \
        ks->threads = 0;                                                                     \
        if (std::is_same<T, __nv_bfloat16>::value && DD == 128 && GG == 4 && kv_pairs) {     \
            ks->decode = reinterpret_cast<const void*>(tc_fp8_kernel<T>());                   \
            ks->warp_bytes = CfgTc::kPipeBytes;                                              \
            ks->rows_per_stage = kMmaRows;                                                   \
            ks->part_heads = 8;                                                              \
            ks->smem_slack = 1024;                                                           \
            ks->max_warps = CfgTc::kPipes;                                                   \
            ks->threads = CfgTc::kThreads;                                                   \
            ks->mma = 3;                                                                     \
        } else if constexpr (DD >= 128 && GG >= 4) {                                         \
            ks->decode = reinterpret_cast<const void*>(decode_fp8_mma_kernel<T, DD>);        \
            ks->warp_bytes = CfgF8<DD>::kWarpBytes;                                          \
            ks->rows_per_stage = kMmaRows;                                                   \
            ks->part_heads = 8;                                                              \
            ks->smem_slack = 1024;                                                           \
            ks->max_warps = CfgF8<DD>::kMaxWarps;                                            \
            ks->mma = 2;                                                                     \
        } else {                                                                             \
            ks->decode = reinterpret_cast<const void*>(decode_kernel<T, DD, GG, kVarFp8>);   \
            ks->warp_bytes = Cfg<T, DD, GG, 1>::kWarpBytes;                                  \
            ks->rows_per_stage = Cfg<T, DD, GG, 1>::kRC;                                     \
            ks->part_heads = GG;                                                             \
            ks->smem_slack = 0;                                                              \
            ks->max_warps = 8;                                                               \
            ks->mma = 0;                                                                     \
        }                                                                                    \
        ks->variant[0] = ks->decode;                                                         \
        ks->variant[1] = ks->variant[2] = ks->variant[3] = nullptr;                          \
        return true;                                                                         \
    }
    PD_CASE(64, 1) PD_CASE(64, 2) PD_CASE(64, 4) PD_CASE(64, 8)
    PD_CASE(128, 1) PD_CASE(128, 2) PD_CASE(128, 4) PD_CASE(128, 8)
    PD_CASE(256, 1) PD_CASE(256, 2) PD_CASE(256, 4) PD_CASE(256, 8)
#undef PD_CASE
    return false;
}

}  // namespace pd
