// Batched decode attention on tensor cores, for 16-bit (f16 / bf16) tiles of
// 4 to 8 q heads per kv head: groups 3..8 (a tile of 3 or 4 heads is padded to
// the 8-head tile) and larger groups cut into tiles of at most 8. Tiles of 1
// or 2 heads and f32 run on CUDA cores (pd_decode.cuh). At group 8 the
// per-byte arithmetic (2 x 8 FMAs per K/V element pair)
// saturates the CUDA cores, while the grouped score tile S = K q^T
// (16 tokens x 8 heads x head_dim) and O^T += V^T P (head_dim x 8 heads x 16
// tokens) are small dense contractions that the mma.sync m16n8k16 units do in
// 24 instructions per 16-token chunk.
//
// Same work partition and walk as the CUDA-core kernel (pd_walk.cuh); the
// differences are:
//  - K and V chunks of 16 rows are staged by 4-D tensor-map TMA
//    (cp.async.bulk.tensor) in 64-column boxes with the 128-byte swizzle, so
//    that ldmatrix reads them without bank conflicts. Rows past the page (or
//    past the cache) are zero-filled by the TMA unit; rows past the valid
//    length in a last page are zeroed in shared memory before P.V.
//  - Scores: A = K rows (ldmatrix), B = q (registers, loaded at a request
//    start), C = 16 x 8 f32. Lane (g = lane/4, c = lane%4) holds tokens g and
//    g+8 of heads 2c and 2c+1, which are also the heads of its P.V
//    accumulator rows, so its softmax state covers exactly its accumulators.
//  - P goes to the P.V tile through movmatrix (transpose of the 8x8 blocks).
//    P is split into a high and a low 16-bit part (p = hi + lo to ~2^-16
//    relative) so that rounding P to 16 bits does not cost accuracy; both
//    parts are multiplied into the same accumulator.
#pragma once

#include <cuda.h>  // CUtensorMap

#include <type_traits>

#include "pd_walk.cuh"

namespace pd {

constexpr int kMmaRows = 16;  // tokens per chunk: the M of the score tile

template <typename T, int D>
struct CfgMma {
    static constexpr int kStages = D <= 128 ? 3 : 2;
    static constexpr int kBoxes = D / 64;               // 64-column (128-byte) boxes per row block
    static constexpr int kBoxBytes = kMmaRows * 128;    // one box: 16 rows x 128 bytes
    static constexpr int kKBytes = kBoxes * kBoxBytes;  // K (and V) bytes of one chunk
    // q is not staged: it is read at a segment start, from L2 (see produce)
    static constexpr int kStageBytes = round_up(2 * kKBytes, 1024);
    static constexpr int kMetaOff = kStages * kStageBytes;
    static constexpr int kBarOff = kMetaOff + kStages * 16;
    static constexpr int kWarpBytes = round_up(kBarOff + kStages * 8, 1024);
    static constexpr int kKSteps = D / 16;  // k steps of the score mma, m tiles of the P.V mma
};

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
    return Elt<T>::pack(lo, hi);
}

template <typename T>
__device__ __forceinline__ float2 unpack_pair(uint32_t w) {
    if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

// kVariant: kVarFused adds the fused append (a.k_new / a.v_new set); kVarNhd
// reads a token-major contiguous cache, whose tensor maps are
// {head_dim, kv heads, rows, slabs} (coordinates kv head and row swap).
template <typename T, int D, int kVariant>
__global__ void __launch_bounds__(256, 1)
    decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kFused = (kVariant & kVarFused) != 0, kNhd = (kVariant & kVarNhd) != 0;
    using C = CfgMma<T, D>;
    constexpr int kS = C::kStages, kKS = C::kKSteps;
    // f16 P would lose small weights to underflow: weights are kept 2^7
    // larger (p <= 2^(kTau+7) < 65504) and the shift is taken out of lse.
    constexpr float kShift = std::is_same<T, __half>::value ? 7.f : 0.f;
    constexpr float kTauM = 8.0f;
    const float kNegInf = -__int_as_float(0x7f800000);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Swizzled TMA boxes want 1024-byte aligned destinations.
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int* s_indptr = reinterpret_cast<int*>(smem);
    int* s_lpl = s_indptr + kTableMax + 1;
    uint8_t* wsm = smem + a.table_bytes + wid * C::kWarpBytes;
    int4* meta = reinterpret_cast<int4*>(wsm + C::kMetaOff);
    const uint32_t wsm_u32 = smem_u32(wsm);
    const uint32_t bar0 = wsm_u32 + C::kBarOff;

    // This warp's unit (see DecodeArgs::unit_transpose).
    const long long gwarp = a.unit_transpose ? (long long)wid * gridDim.x + blockIdx.x
                                             : (long long)blockIdx.x * nwarps + wid;
    const long long ppw = a.pos_per_warp;
    const long long p0 = gwarp * ppw;
    const long long pend = min(p0 + ppw - a.tail, a.total_pos);  // the head of share gwarp
    long long unit = a.tail ? (1 + a.tail_pieces) * gwarp : gwarp;  // unit of the chunks being produced
    bool tails_left = a.tail != 0;
    TailClaim tclaim;
    Walk<kFused> walk(a, s_indptr, s_lpl, p0, pend, lane);
    const int first_page = walk.prefetch_first();
    const int GT = a.heads_per_tile;
    if (lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }

    const uint64_t policy = l2_evict_first_policy();
    // Paged pools of pages of at most 16 rows, without the fused append: chunk
    // s of this warp is position p0 + s while those positions belong to
    // requests, so the first stages' copies go out as soon as their page ids
    // are known, before the table is staged (they take the place of the
    // first-slab L2 prefetch). A bad page id is an out-of-range coordinate,
    // which reads zeros; its chunk has no rows.
    // Positions outside [indptr[0], indptr[batch]) (entries of `indices` that
    // no request lists) have no chunk, so the early copies stop at the first
    // such position: every position before it is one chunk, in order.
    const bool early_ok = !kFused && !kNhd && !a.contiguous && a.page_size <= kMmaRows;
    const int cov_lo = early_ok ? __ldg(a.indptr) : 0;
    const int cov_hi = early_ok ? __ldg(a.indptr + a.batch) : 0;
    int n_early = 0;
    walk.stage_table(s_indptr, s_lpl, [&] {
        if (lane == 0) {
            for (int s = 0; s < kS; ++s) mbar_init(bar0 + 8 * s, 1);
            fence_mbar_init();
        }
        if (early_ok) {
            const long long lim = min((long long)kS, max(pend - p0, 0LL));
            while (n_early < lim) {
                const long long i = (p0 + n_early) % a.n_pos;
                if (i < cov_lo || i >= cov_hi) break;
                ++n_early;
            }
        }
        if (n_early == 0) {
            walk.template prefetch_first_slabs<kNhd>(first_page, kS, size_t(D) * sizeof(T));
            return;
        }
        for (int s = 0; s < n_early; ++s) {
            const int pg = __shfl_sync(kFull, first_page, s);
            if (lane == 0) {
                const int kh = int((p0 + s) / a.n_pos) / a.head_tiles;
                const uint32_t bar = bar0 + 8 * s;
                const uint32_t st = wsm_u32 + s * C::kStageBytes;
                // a.test_extra_tx (test-only, normally 0): see the first produce calls below
                mbar_arrive_expect_tx(bar, 2u * C::kKBytes + ((s == 0 && gwarp == 0) ? uint32_t(a.test_extra_tx) : 0u));
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx) {
                    tma_load_4d(st + bx * C::kBoxBytes, &tmk, bx * 64, 0, kh, pg, bar, policy);
                    tma_load_4d(st + C::kKBytes + bx * C::kBoxBytes, &tmv, bx * 64, 0, kh, pg, bar, policy);
                }
            }
        }
    });
    __syncthreads();  // the only block-wide barrier
    launch_dependents();
    if (p0 >= pend && !tails_left) return;  // with tails a warp without a head may still take some
    walk.build(p0, first_page);

    const size_t row_bytes = size_t(D) * sizeof(T);
    // issued: the chunk's copies went out early (see n_early); only its
    // description is written here.
    auto produce = [&](int slot, uint32_t extra_tx, bool issued) {
        Chunk ck;
        // When this warp's range is done, it moves on to tail pieces (claimed ahead).
        const bool have = next_with_tails<kMmaRows>(a, walk, tclaim, &tails_left, &unit, kS, lane, &ck);
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t st = wsm_u32 + slot * C::kStageBytes;
        if constexpr (kFused) {
            if (have && (ck.flags & kAppendRow)) write_new_row<kNhd>(a, ck, lane, row_bytes);
        }
        if (lane != 0) return;
        if (!have) {
            meta[slot] = make_int4(0, kEndOfWork, 0, 0);
            mbar_arrive(bar);
            return;
        }
        meta[slot] = make_int4(ck.rows, ck.flags, ck.qrow, ck.seg + int(unit));  // .w: partial slot
        // A box always lands whole (rows outside the tensor are zero-filled).
        const uint32_t kv_bytes = ck.rows > 0 ? uint32_t(C::kKBytes) : 0u;
        // A segment's q rows are pulled into L2 with its first chunk; the
        // consumer reads them from there when it reaches that chunk.
        if (ck.flags & kSegStart)
            bulk_prefetch_l2(static_cast<const uint8_t*>(a.q) + size_t(ck.qrow) * row_bytes, uint32_t(GT * row_bytes));
        if (issued) return;
        const uint32_t total = 2 * kv_bytes;
        if (total == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, total + extra_tx);
        if (kv_bytes) {
            const int c1 = kNhd ? ck.kh : ck.row0, c2 = kNhd ? ck.row0 : ck.kh;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
                tma_load_4d(st + bx * C::kBoxBytes, &tmk, bx * 64, c1, c2, ck.slab, bar, policy);
                tma_load_4d(st + C::kKBytes + bx * C::kBoxBytes, &tmv, bx * 64, c1, c2, ck.slab, bar, policy);
            }
        }
    };

    // ---- consumer state: lane (g, c) owns tokens g, g+8 and heads 2c, 2c+1
    const int g = lane >> 2, c = lane & 3;
    uint32_t qf[kKS][2];  // score-mma B fragments: q[head g][16kk + 2c (+8) ...]
    float acc[kKS][4];    // P.V accumulators: o^T[16mt + g (+8)][head 2c (+1)]
    float m0, m1, l0, l1;  // reference max and weight sum of heads 2c, 2c+1 (this lane's tokens)
    auto reset_state = [&]() {
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        m0 = m1 = kNegInf;
        l0 = l1 = 0.f;
    };
    reset_state();
#pragma unroll
    for (int kk = 0; kk < kKS; ++kk) qf[kk][0] = qf[kk][1] = 0u;

    auto finalize = [&](int4 m) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        const int qrow = m.z;
        const int h0 = 2 * c, h1 = 2 * c + 1;
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const float lse0 = l0 > 0.f ? m0 - kShift + log2f(l0) : kNegInf;
        const float lse1 = l1 > 0.f ? m1 - kShift + log2f(l1) : kNegInf;
        if (m.y & kSegComplete) {
            T* o0 = static_cast<T*>(a.o) + (size_t(qrow) + h0) * D;
            T* o1 = o0 + D;
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                const int d = 16 * mt + g;
                if (h0 < GT) {
                    o0[d] = T(acc[mt][0] * inv0);
                    o0[d + 8] = T(acc[mt][2] * inv0);
                }
                if (h1 < GT) {
                    o1[d] = T(acc[mt][1] * inv1);
                    o1[d + 8] = T(acc[mt][3] * inv1);
                }
            }
            if (g == 0 && a.lse != nullptr) {
                if (h0 < GT) a.lse[size_t(qrow) + h0] = lse0 == kNegInf ? kNegInf : lse0 * kLn2;
                if (h1 < GT) a.lse[size_t(qrow) + h1] = lse1 == kNegInf ? kNegInf : lse1 * kLn2;
            }
        } else {
            const long long slot = m.w;
            float* p0r = a.part_o + (size_t(slot) * 8 + h0) * D;
            float* p1r = p0r + D;
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                const int d = 16 * mt + g;
                if (h0 < GT) {
                    p0r[d] = acc[mt][0] * inv0;
                    p0r[d + 8] = acc[mt][2] * inv0;
                }
                if (h1 < GT) {
                    p1r[d] = acc[mt][1] * inv1;
                    p1r[d + 8] = acc[mt][3] * inv1;
                }
            }
            if (g == 0) {
                if (h0 < GT) a.part_lse[size_t(slot) * 8 + h0] = lse0;
                if (h1 < GT) a.part_lse[size_t(slot) * 8 + h1] = lse1;
            }
        }
        reset_state();
    };

    auto consume = [&](int slot, int4 m) {
        const uint32_t ks = wsm_u32 + slot * C::kStageBytes;
        const uint32_t vs = ks + C::kKBytes;
        uint8_t* stp = wsm + slot * C::kStageBytes;
        if (m.y & kSegStart) {
            const uint8_t* qb = static_cast<const uint8_t*>(a.q) + (size_t(m.z) + g) * row_bytes;
#pragma unroll
            for (int kk = 0; kk < kKS; ++kk) {
                qf[kk][0] = g < GT ? __ldg(reinterpret_cast<const uint32_t*>(qb + (16 * kk + 2 * c) * 2)) : 0u;
                qf[kk][1] = g < GT ? __ldg(reinterpret_cast<const uint32_t*>(qb + (16 * kk + 2 * c + 8) * 2)) : 0u;
            }
        }
        const int rows = m.x;
        if (rows < kMmaRows) {
            // V rows past the valid length may hold anything (the page's tail):
            // zero them so that their zero weights give zero products.
            const int n = (kMmaRows - rows) * C::kBoxes * 8;
            for (int idx = lane; idx < n; idx += 32) {
                const int r = rows + idx / (C::kBoxes * 8), rem = idx % (C::kBoxes * 8);
                *reinterpret_cast<uint4*>(stp + C::kKBytes + (rem >> 3) * C::kBoxBytes + r * 128 + (rem & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        // scores S[16 tokens][8 heads]
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int r = lane & 15;
#pragma unroll
            for (int kk = 0; kk < kKS; ++kk) {
                const int ch = ((kk & 3) << 1) + (lane >> 4);
                uint32_t af[4];
                ldsm_x4(ks + (kk >> 2) * C::kBoxBytes + r * 128 + ((ch ^ (r & 7)) << 4), af);
                mma_16816<T>(sc, af, qf[kk][0], qf[kk][1]);
            }
        }
        float x0 = g < rows ? sc[0] * a.q_scale : kNegInf;
        float x1 = g < rows ? sc[1] * a.q_scale : kNegInf;
        float x2 = g + 8 < rows ? sc[2] * a.q_scale : kNegInf;
        float x3 = g + 8 < rows ? sc[3] * a.q_scale : kNegInf;
        const bool need = x0 > m0 + kTauM || x2 > m0 + kTauM || x1 > m1 + kTauM || x3 > m1 + kTauM;
        if (__any_sync(kFull, need)) {
            float c0 = fmaxf(x0, x2), c1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                c0 = fmaxf(c0, __shfl_xor_sync(kFull, c0, off));
                c1 = fmaxf(c1, __shfl_xor_sync(kFull, c1, off));
            }
            const float n0 = fmaxf(m0, c0), n1 = fmaxf(m1, c1);
            const float al0 = n0 == kNegInf ? 1.f : ex2(m0 - n0), al1 = n1 == kNegInf ? 1.f : ex2(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                acc[mt][0] *= al0;
                acc[mt][2] *= al0;
                acc[mt][1] *= al1;
                acc[mt][3] *= al1;
            }
        }
        const float p0 = x0 == kNegInf ? 0.f : ex2(x0 - m0 + kShift);
        const float p1 = x1 == kNegInf ? 0.f : ex2(x1 - m1 + kShift);
        const float p2 = x2 == kNegInf ? 0.f : ex2(x2 - m0 + kShift);
        const float p3 = x3 == kNegInf ? 0.f : ex2(x3 - m1 + kShift);
        l0 += p0 + p2;
        l1 += p1 + p3;
        const uint32_t h01 = pack_pair<T>(p0, p1), h23 = pack_pair<T>(p2, p3);
        const float2 r01 = unpack_pair<T>(h01), r23 = unpack_pair<T>(h23);
        const uint32_t l01 = pack_pair<T>(p0 - r01.x, p1 - r01.y), l23 = pack_pair<T>(p2 - r23.x, p3 - r23.y);
        const uint32_t bh0 = movm_trans(h01), bh1 = movm_trans(h23);
        const uint32_t bl0 = movm_trans(l01), bl1 = movm_trans(l23);
        // O^T[head_dim][8 heads] += V^T[head_dim][16 tokens] P[16 tokens][8 heads]
        {
            const int mi = lane >> 3;
            const int tok = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                const int ch = ((mt & 3) << 1) + (mi & 1);
                uint32_t af[4];
                ldsm_x4_trans(vs + (mt >> 2) * C::kBoxBytes + tok * 128 + ((ch ^ (tok & 7)) << 4), af);
                mma_16816<T>(acc[mt], af, bh0, bh1);
                mma_16816<T>(acc[mt], af, bl0, bl1);
            }
        }
        if (m.y & kSegEnd) finalize(m);
    };

    // a.test_extra_tx (test-only, normally 0): warp 0's first stage expects
    // bytes that never arrive, so that its bounded wait runs out.
#pragma unroll 1
    for (int s = 0; s < kS; ++s) produce(s, (s == 0 && gwarp == 0) ? uint32_t(a.test_extra_tx) : 0u, s < n_early);
#pragma unroll 1
    for (int it = 0;; ++it) {
        const int slot = it % kS;
        const uint32_t parity = uint32_t(it / kS) & 1u;
        if (!mbar_wait_bounded(bar0 + 8 * slot, parity)) {
            if (lane == 0) atomicOr(a.flags, kFlagTimeout);
            for (int s = 1; s < kS; ++s) {
                const int it2 = it + s;
                mbar_wait_bounded(bar0 + 8 * (it2 % kS), uint32_t(it2 / kS) & 1u);
            }
            break;
        }
        const int4 m = meta[slot];
        if (m.y & kEndOfWork) break;
        consume(slot, m);
        __syncwarp();
        produce(slot, 0u, false);
    }
    tails_finished(a, nwarps, lane);
}

}  // namespace pd
