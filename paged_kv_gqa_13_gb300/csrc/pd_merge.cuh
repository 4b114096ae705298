// Merge of split attention states: the kernel that combines the decode's
// partial (o, lse) results, and the standalone merge of caller-supplied parts.
#pragma once

#include "pd_walk.cuh"

namespace pd {

// Weighted sum of partial rows, parts taken in index order: lane c of each
// group of 32 parts computes its part's weight 2^(lse_c - L); the weights are
// broadcast with shuffles and every lane accumulates its kPer columns. Rows
// are loaded in rounds of kRound (the caller's register budget); the first
// round is requested together with the lse values, so up to kRound parts take
// one round trip and every further kRound parts one more.
template <int kPer, int kRoundMax = 16, class LseAt, class RowAt>
__device__ __forceinline__ float merge_rows(int parts, LseAt lse_at, RowAt row_at, float* acc) {
    const float kNegInf = -__int_as_float(0x7f800000);
    const int lane = threadIdx.x & 31;
    constexpr int kRound = (64 / kPer) < kRoundMax ? (64 / kPer) : kRoundMax;  // divides 32
    static_assert(32 % kRound == 0, "a round never straddles two groups of 32 parts");
    float rows[kRound][kPer];
    auto load_round = [&](int base) {
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            if (base + j < parts) {
                const float* po = row_at(base + j) + lane * kPer;
#pragma unroll
                for (int e = 0; e < kPer; e += 2) {
                    const float2 t = *reinterpret_cast<const float2*>(po + e);
                    rows[j][e] = t.x;
                    rows[j][e + 1] = t.y;
                }
            }
        }
    };
    const float mine = lane < parts ? lse_at(lane) : kNegInf;
    load_round(0);
    float M = mine;
    for (int cp = lane + 32; cp < parts; cp += 32) M = fmaxf(M, lse_at(cp));
    M = warp_max(M);
    if (M == kNegInf) return kNegInf;
    float S = lane < parts ? ex2(mine - M) : 0.f;
    for (int cp = lane + 32; cp < parts; cp += 32) S += ex2(lse_at(cp) - M);
    S = warp_sum(S);
    const float L = M + log2f(S);
    float w_mine = lane < parts ? ex2(mine - L) : 0.f;  // weight of part (base & ~31) + lane
    for (int base = 0; base < parts; base += kRound) {
        if (base > 0) {
            if ((base & 31) == 0) w_mine = base + lane < parts ? ex2(lse_at(base + lane) - L) : 0.f;
            load_round(base);
        }
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            const float w = __shfl_sync(kFull, w_mine, (base + j) & 31);
            if (base + j < parts) {
#pragma unroll
                for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, rows[j][e], acc[e]);
            }
        }
    }
    return L;
}

template <typename T, int kPer>
__device__ __forceinline__ void store_row(T* orow, const float* acc) {
    const int lane = threadIdx.x & 31;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<float2*>(reinterpret_cast<float*>(orow) + lane * kPer + e) = make_float2(acc[e], acc[e + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<uint32_t*>(orow + lane * kPer + e) = Elt<T>::pack(acc[e], acc[e + 1]);
    }
}

// One warp per (request, kv head, head tile, q head): combine the partial
// results the decode warps wrote for a request split across warps, in warp
// order; write zeros / -inf for requests with no pages. Everything that does
// not depend on the decode's output (the page table, empty requests) is done
// before waiting for the decode grid.
// Its grid follows the decode with one warp per (segment, head). Registers
// are held to 85 per thread (rounds of 8 parts, 4 at head_dim 256) so that 6
// blocks fit per SM and the warps that remain after the decode run in few
// waves. kWide (for grids that fit one wave at 4 blocks per SM): rounds of 16
// parts (8 at 256), so that requests split over up to 16 units take one
// round trip.
template <typename T, int D, bool kWide = false>
__global__ void __launch_bounds__(128, kWide ? 4 : 6) merge_partials_kernel(const MergeArgs a) {
    constexpr int kPer = D / 32;  // elements per lane
    const float kNegInf = -__int_as_float(0x7f800000);
    const int lane = threadIdx.x & 31;
    const long long pair = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long segments = (long long)a.head_tiles * a.num_kv_heads * a.batch;
    if (pair >= segments * a.heads_per_tile) return;
    const int h = int(pair % a.heads_per_tile);
    const long long s = pair / a.heads_per_tile;
    const int b = int(s % a.batch), sh = int(s / a.batch);
    const int kh = sh / a.head_tiles, ht = sh % a.head_tiles;
    const int head = kh * a.group + ht * a.heads_per_tile + h;
    int lo, hi;
    if (a.contiguous) {
        request_range(b, a.n_pos, true, a.npv, 0, 0, &lo, &hi);
    } else {
        const int r0 = __ldg(a.indptr + b), r1 = __ldg(a.indptr + b + 1);
        if (sh == 0 && h == 0 && lane == 0 && (r0 < 0 || r1 < r0 || r1 > a.n_pos))
            atomicOr(a.flags, kFlagBadIndptr);
        request_range(b, a.n_pos, false, 0, r0, r1, &lo, &hi);
    }
    T* orow = static_cast<T*>(a.o) + (size_t(b) * a.num_qo_heads + head) * D;
    float* lse_out = a.lse ? a.lse + size_t(b) * a.num_qo_heads + head : nullptr;
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float L = kNegInf;
    if (a.append && hi <= lo && sh == 0 && h == 0 && lane == 0) atomicOr(a.flags, kFlagBadIndptr);
    if (hi > lo) {
        const long long first = unit_of((long long)sh * a.n_pos + lo, a.pos_per_warp, a.tail, a.tail_pieces);
        const long long last = unit_of((long long)sh * a.n_pos + hi - 1, a.pos_per_warp, a.tail, a.tail_pieces);
        if (first == last) return;  // one warp held the whole request and wrote it
        grid_dependency_wait();     // the decode kernel's partials are complete and visible
        const int parts = int(last - first + 1);
        const long long slot0 = (first + s) * a.G + h;  // slot of part c: (first + c + s) * G + h
        L = merge_rows<kPer, (D <= 128 ? 8 : 4) * (kWide ? 2 : 1)>(
            parts, [&](int cp) { return a.part_lse[slot0 + (long long)cp * a.G]; },
            [&](int cp) { return a.part_o + size_t(slot0 + (long long)cp * a.G) * D; }, acc);
    }
    store_row<T, kPer>(orow, acc);
    if (lse_out && lane == 0) *lse_out = (L == kNegInf) ? kNegInf : L * kLn2;
}

// Standalone merge of caller-supplied parts (natural-log lse), one warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_states_kernel(const float* o_parts, const float* lse_parts,
                                                            int num_parts, int num_rows, void* o, float* lse) {
    constexpr int kPer = D / 32;
    const float kNegInf = -__int_as_float(0x7f800000);
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= num_rows) return;
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    const float L = merge_rows<kPer>(
        num_parts, [&](int cp) { return lse_parts[size_t(cp) * num_rows + row] * kLog2e; },
        [&](int cp) { return o_parts + (size_t(cp) * num_rows + row) * D; }, acc);
    store_row<T, kPer>(static_cast<T*>(o) + size_t(row) * D, acc);
    if (lse && lane == 0) lse[row] = (L == kNegInf) ? kNegInf : L * kLn2;
}

}  // namespace pd
