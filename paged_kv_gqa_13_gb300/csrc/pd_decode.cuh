// Batched decode attention over a paged (or contiguous) KV cache on CUDA
// cores: the kernel for f32 at every group, for 16-bit tiles of 1 or 2 q
// heads per kv head (16-bit tiles of 4 to 8 heads run on the tensor-core
// kernel, pd_decode_mma.cuh), and, as a variant, for E4M3 pools outside the
// E4M3 tensor-core kernel's shapes.
//
// Work decomposition (see pd_walk.cuh). All positions of the call are cut into
// equal contiguous ranges, one per warp of a grid that fills every SM. A warp
// therefore streams ~total_pos/warps page slices whatever the length mix: a
// long request is split over several warps (split-KV), many short ones share
// a warp. Where a warp's range covers a request's whole page list the warp
// writes o and lse itself; otherwise it writes a normalised partial (o, lse)
// into workspace slot (unit + segment), and merge_partials_kernel combines
// the partials in unit order.
//
// Inside a warp. The warp runs its own kStages-deep ring in shared memory.
// Lane 0 issues 1-D bulk async copies (cp.async.bulk) of K and V page slices
// -- in the HND layout rows [r0, r1) of one (page, kv head) are one
// contiguous block; the token-major (NHD) variant uses tensor-map boxes
// instead -- plus, at the start of a request, the group's q rows.
// Completion is counted in bytes on the stage's mbarrier. While one stage is
// being consumed, the next ones are in flight.
//
// Arithmetic (f32). Lane (row group rg, column c) holds EPL elements of the
// head dimension for every q head of the group. For a round of RR rows it
// forms the group's partial dot products for those rows with packed f32x2
// FMAs, then a reduce-scatter over the L lanes of the row group leaves each
// lane with a few complete scores. Softmax runs in log2 units (q is
// pre-scaled by sm_scale*log2 e) against a per-head reference maximum m that
// only moves when a score exceeds it by more than kTau; a move rescales the
// accumulators. P is broadcast through shared memory and every lane adds
// p * v into its accumulators for its columns. K and V bytes are read from
// HBM once for the whole group.
#pragma once

#include "pd_walk.cuh"

namespace pd {

constexpr int kStages = 3;
constexpr int kChunkBytes = 4096;  // K bytes of one stage (V the same)
constexpr float kTau = 8.0f;       // reference max slack, log2 units: p <= 2^kTau

// KvEsz: bytes per K/V element (sizeof(T), or 1 for E4M3 pools). q, o and
// the lane-to-column map follow T either way.
template <typename T, int D, int G, int KvEsz = int(sizeof(T))>
struct Cfg {
    static constexpr int kEsz = int(sizeof(T));
    static constexpr int kVec = 16 / kEsz;           // elements per 16-byte vector
    static constexpr int kEpl = (G <= 4) ? 16 : 8;   // elements per lane per row
    static constexpr int kNvec = kEpl / kVec;        // vectors per lane per row
    static constexpr int kL = D / kEpl;              // lanes per row
    static constexpr int kRW = 32 / kL;              // rows side by side in a warp
    static constexpr int kRowBytes = D * kEsz;            // q / o row
    static constexpr int kKvRowBytes = D * KvEsz;         // K / V row
    static constexpr int kRC = kChunkBytes / kKvRowBytes;  // rows per stage
    static constexpr int kRR0 = (16 / G) > 0 ? (16 / G) : 1;
    static constexpr int kRR = kRR0 < (kRC / kRW) ? kRR0 : (kRC / kRW);  // rows per row group per round
    static constexpr int kRounds = kRC / (kRW * kRR);
    static constexpr int kV = kRR * G;               // partial sums per lane per round
    static constexpr int kVF = kV >= kL ? kV / kL : 1;  // complete scores per lane after the reduction
    static constexpr int kQBytes = G * D * kEsz;
    static constexpr int kStageBytes = round_up(2 * kChunkBytes + kQBytes, 128);
    static constexpr int kMetaOff = kStages * kStageBytes;
    static constexpr int kBarOff = kMetaOff + kStages * 16;
    static constexpr int kPbufOff = round_up(kBarOff + kStages * 8, 16);  // read as float4
    static constexpr int kWarpBytes = round_up(kPbufOff + kRW * kV * 4, 128);
    static_assert(kL >= 1 && kL <= 32 && (kL & (kL - 1)) == 0, "lanes per row");
    static_assert(kEpl % kVec == 0, "whole vectors per lane");
    static_assert(kRC >= kRW && kRC % (kRW * kRR) == 0, "rows per stage");
};

// kVariant: kVarFused adds the fused append (a.k_new / a.v_new set); kVarNhd
// reads a token-major contiguous cache through the tensor maps tmk / tmv
// ({head_dim, kv heads, valid rows, requests}, boxes of kRC rows of one kv
// head, unswizzled, rows past the valid length zero-filled); the other
// variants do not read the maps.
template <typename T, int D, int G, int kVariant>
__global__ void __launch_bounds__(256, 1)
    decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kFused = (kVariant & kVarFused) != 0, kNhd = (kVariant & kVarNhd) != 0;
    constexpr bool kFp8 = (kVariant & kVarFp8) != 0;
    static_assert(!kFp8 || (sizeof(T) == 2 && !kFused && !kNhd), "E4M3 pools: 16-bit q / o, paged, no fused append");
    using C = Cfg<T, D, G, kFp8 ? 1 : int(sizeof(T))>;
    using E = Elt<T>;
    constexpr int kL = C::kL, kRW = C::kRW, kRR = C::kRR, kV = C::kV, kVF = C::kVF;
    constexpr int kVec = C::kVec, kNvec = C::kNvec, kEpl = C::kEpl, kRC = C::kRC;
    const float kNegInf = -__int_as_float(0x7f800000);

    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int* s_indptr = reinterpret_cast<int*>(smem);
    int* s_lpl = s_indptr + kTableMax + 1;
    uint8_t* wsm = smem + a.table_bytes + wid * C::kWarpBytes;
    int4* meta = reinterpret_cast<int4*>(wsm + C::kMetaOff);
    const uint32_t bar0 = smem_u32(wsm + C::kBarOff);
    float* pbuf = reinterpret_cast<float*>(wsm + C::kPbufOff);

    // This warp's range of positions; the page ids of its first two windows
    // are requested before the set-up so that their latency overlaps it.
    // This warp's unit (see DecodeArgs::unit_transpose).
    const long long gwarp = a.unit_transpose ? (long long)wid * gridDim.x + blockIdx.x
                                             : (long long)blockIdx.x * nwarps + wid;
    const long long p0 = gwarp * a.pos_per_warp;
    const long long pend = min(p0 + a.pos_per_warp - a.tail, a.total_pos);  // the head of share gwarp
    long long unit = a.tail ? (1 + a.tail_pieces) * gwarp : gwarp;           // unit of the chunks produced
    bool tails_left = a.tail != 0;
    TailClaim tclaim;
    Walk<kFused> walk(a, s_indptr, s_lpl, p0, pend, lane);
    const int first_page = walk.prefetch_first();
    const int GT = a.heads_per_tile;
    if constexpr (kNhd) {
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
    }

    // ---- set-up: stage the page table, zero the ring, init the barriers
    walk.stage_table(s_indptr, s_lpl, [&] {
        // Rows of a stage that no copy fills must still hold finite numbers,
        // since their (zero) softmax weight multiplies them.
        for (int off = lane * 16; off < kStages * C::kStageBytes; off += 32 * 16)
            *reinterpret_cast<uint4*>(wsm + off) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
            fence_mbar_init();
        }
        walk.template prefetch_first_slabs<kNhd>(first_page, kStages, size_t(C::kKvRowBytes));
    });
    __syncthreads();  // the only block-wide barrier: warps are independent from here on
    // Let the merge kernel be scheduled now; it waits for this grid before it
    // reads any partial result.
    launch_dependents();
    if (p0 >= pend && !tails_left) return;  // with tails a warp without a head may still take some
    walk.build(p0, first_page);

    const uint64_t policy = l2_evict_first_policy();
    const size_t row_bytes = size_t(C::kRowBytes);       // q
    const size_t kv_row_bytes = size_t(C::kKvRowBytes);  // K, V
    // Emit the next chunk into `slot` (whole warp; lane 0 issues the copies).
    auto produce = [&](int slot, uint32_t extra_tx) {
        Chunk ck;
        // When this warp's range is done, it moves on to tail pieces (claimed ahead).
        const bool have = next_with_tails<kRC>(a, walk, tclaim, &tails_left, &unit, kStages, lane, &ck);
        const uint32_t bar = bar0 + 8 * slot;
        uint8_t* st = wsm + slot * C::kStageBytes;
        if constexpr (kFused) {
            if (have && (ck.flags & kAppendRow)) write_new_row<kNhd>(a, ck, lane, kv_row_bytes);
        }
        if (lane != 0) return;
        if (!have) {
            meta[slot] = make_int4(0, kEndOfWork, 0, 0);
            mbar_arrive(bar);
            return;
        }
        meta[slot] = make_int4(ck.rows, ck.flags, ck.qrow, ck.seg + int(unit));  // .w: partial slot
        // An NHD box lands whole: kRC rows, those past the valid length as zeros.
        const uint32_t kv_bytes =
            kNhd ? (ck.rows > 0 ? uint32_t(kChunkBytes) : 0u) : uint32_t(ck.rows) * uint32_t(kv_row_bytes);
        const uint32_t q_bytes = (ck.flags & kSegStart) ? uint32_t(GT * C::kRowBytes) : 0u;
        const uint32_t total = 2 * kv_bytes + q_bytes;
        if (total == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, total + extra_tx);
        if (kv_bytes) {
            if constexpr (kNhd) {
                tma_load_4d(smem_u32(st), &tmk, 0, ck.kh, ck.row0, ck.slab, bar, policy);
                tma_load_4d(smem_u32(st + kChunkBytes), &tmv, 0, ck.kh, ck.row0, ck.slab, bar, policy);
            } else {
                const size_t off = kv_row<false>(a, ck.slab, ck.kh, ck.row0) * kv_row_bytes;
                bulk_g2s(smem_u32(st), static_cast<const uint8_t*>(a.k) + off, kv_bytes, bar, policy);
                bulk_g2s(smem_u32(st + kChunkBytes), static_cast<const uint8_t*>(a.v) + off, kv_bytes, bar, policy);
            }
        }
        if (q_bytes)
            bulk_g2s(smem_u32(st + 2 * kChunkBytes), static_cast<const uint8_t*>(a.q) + size_t(ck.qrow) * row_bytes,
                     q_bytes, bar);
    };

    // ---- consumer state
    const int c = lane % kL;  // column within the row group
    const int rg = lane / kL;  // row group
    using RS = ReduceScatter<kV, kL / 2>;
    int hj[kVF], rj[kVF], ij[kVF];
#pragma unroll
    for (int j = 0; j < kVF; ++j) {
        ij[j] = RS::index(j, lane);
        hj[j] = ij[j] % G;
        rj[j] = ij[j] / G;
    }
    // When a round has fewer values than lanes, groups of lanes hold copies of
    // one value; only the first lane of each group counts it into the sum.
    const bool primary = (kV >= kL) || ((c & ((kL >= kV ? kL / kV : 1) - 1)) == 0);

    // q and the accumulators are kept as float2 pairs of adjacent columns so
    // that the dot products and the P.V update use packed f32x2 FMAs.
    constexpr int kEp2 = kEpl / 2;
    float2 qf[G][kEp2];
    float2 acc[G][kEp2];
    float mref[G];
    float mmy[kVF], lmy[kVF];
    auto reset_state = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mref[h] = kNegInf;
#pragma unroll
            for (int e = 0; e < kEp2; ++e) acc[h][e] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kVF; ++j) mmy[j] = kNegInf, lmy[j] = 0.f;
    };
    auto pick = [&](const float* arr, int h) -> float {
        float r = arr[0];
#pragma unroll
        for (int x = 1; x < G; ++x) r = (h == x) ? arr[x] : r;
        return r;
    };
    reset_state();

    // End of this warp's share of a request: sum the row groups' accumulators
    // (a reduce-scatter, so each lane ends up owning a share of the columns
    // of the group's heads), then write o and lse, or the normalised partial.
    using RSR = ReduceScatter2<G * kEp2, 16, kL>;
    constexpr int kOwn = (kRW > 1) ? G * kEp2 / kRW : G * kEp2;  // float2 values a lane writes
    auto finalize = [&](int4 m) {
        float lh[G], inv[G];
        // E4M3 pools: the V scale of this kv head is applied once, here.
        const float vsc = kFp8 ? __ldg(a.v_scale + (m.z % a.num_qo_heads) / a.group) : 1.0f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kVF; ++j) s += (primary && hj[j] == h) ? lmy[j] : 0.f;
            lh[h] = warp_sum(s);
            inv[h] = lh[h] > 0.f ? vsc / lh[h] : 0.f;
        }
        float2* flat = &acc[0][0];
        RSR::run(flat, lane);
        const int qrow = m.z;  // first q / o row of the group
        const bool complete = (m.y & kSegComplete) != 0;
        const long long slot = m.w;
#pragma unroll
        for (int j = 0; j < kOwn; ++j) {
            const int x = RSR::index(j, lane);
            const int h = x / kEp2, e = 2 * (x % kEp2);
            if (h >= GT) continue;
            const int d = ((e / kVec) * kL + c) * kVec + (e % kVec);
            const float iv = pick(inv, h);
            const float2 val = make_float2(flat[j].x * iv, flat[j].y * iv);
            if (complete) {
                T* orow = static_cast<T*>(a.o) + (size_t(qrow) + h) * D;
                if constexpr (sizeof(T) == 4) {
                    *reinterpret_cast<float2*>(orow + d) = val;
                } else {
                    *reinterpret_cast<uint32_t*>(orow + d) = E::pack(val.x, val.y);
                }
            } else {
                *reinterpret_cast<float2*>(a.part_o + (size_t(slot) * G + h) * D + d) = val;
            }
        }
        if (lane < GT) {
            const float l = pick(lh, lane), mr = pick(mref, lane);
            if (complete) {
                if (a.lse != nullptr) a.lse[size_t(qrow) + lane] = l > 0.f ? (mr + log2f(l)) * kLn2 : kNegInf;
            } else {
                a.part_lse[size_t(slot) * G + lane] = l > 0.f ? mr + log2f(l) : kNegInf;
            }
        }
        reset_state();
    };

    auto consume = [&](int slot, int4 m) {
        const uint8_t* kb = wsm + slot * C::kStageBytes;
        const uint8_t* vb = kb + kChunkBytes;
        if (m.y & kSegStart) {
            const uint8_t* qb = kb + 2 * kChunkBytes;
            // E4M3 pools: the K scale of this kv head folds into q.
            const float qs = kFp8 ? a.q_scale * __ldg(a.k_scale + (m.z % a.num_qo_heads) / a.group) : a.q_scale;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int nv = 0; nv < kNvec; ++nv) {
                    float f[kVec];
                    if (h < GT) {
                        E::to_f32(*reinterpret_cast<const uint4*>(qb + h * C::kRowBytes + (nv * kL + c) * 16), f);
                    } else {
#pragma unroll
                        for (int e = 0; e < kVec; ++e) f[e] = 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < kVec / 2; ++e)
                        qf[h][nv * kVec / 2 + e] = make_float2(f[2 * e] * qs, f[2 * e + 1] * qs);
                }
        }
        const int rows = m.x;
#pragma unroll
        for (int rd = 0; rd < C::kRounds; ++rd) {
            const int r0 = rd * kRW * kRR;
            if (r0 >= rows) break;
            // scores: partial dot products of this lane's columns, even and odd
            // columns in the two halves of a float2
            float2 part2[kV];
#pragma unroll
            for (int x = 0; x < kV; ++x) part2[x] = make_float2(0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < kRR; ++rr) {
                const int r = r0 + rr * kRW + rg;
#pragma unroll
                for (int nv = 0; nv < kNvec; ++nv) {
                    float f[kVec];
                    if constexpr (kFp8)
                        e4m3x8_to_f32(*reinterpret_cast<const uint2*>(kb + r * C::kKvRowBytes + (nv * kL + c) * 8), f);
                    else
                        E::to_f32(*reinterpret_cast<const uint4*>(kb + r * C::kKvRowBytes + (nv * kL + c) * 16), f);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < kVec / 2; ++e)
                            part2[rr * G + h] = __ffma2_rn(qf[h][nv * kVec / 2 + e],
                                                           make_float2(f[2 * e], f[2 * e + 1]), part2[rr * G + h]);
                }
            }
            float part[kV];
#pragma unroll
            for (int x = 0; x < kV; ++x) part[x] = part2[x].x + part2[x].y;
            RS::run(part, lane);
            // softmax against the reference max
            float x[kVF];
            bool need = false;
#pragma unroll
            for (int j = 0; j < kVF; ++j) {
                const int r = r0 + rj[j] * kRW + rg;
                x[j] = (r < rows) ? part[j] : kNegInf;
                need |= x[j] > mmy[j] + kTau;
            }
            if (__any_sync(kFull, need)) {
                float alpha[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float mh = kNegInf;
#pragma unroll
                    for (int j = 0; j < kVF; ++j) mh = (hj[j] == h) ? fmaxf(mh, x[j]) : mh;
                    mh = warp_max(mh);
                    const float mn = fmaxf(mref[h], mh);
                    alpha[h] = (mn == kNegInf) ? 1.f : ex2(mref[h] - mn);
                    mref[h] = mn;
                    const float2 al2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
                    for (int e = 0; e < kEp2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], al2);
                }
#pragma unroll
                for (int j = 0; j < kVF; ++j) {
                    lmy[j] *= pick(alpha, hj[j]);
                    mmy[j] = pick(mref, hj[j]);
                }
            }
            float p[kVF];
#pragma unroll
            for (int j = 0; j < kVF; ++j) {
                p[j] = (x[j] == kNegInf) ? 0.f : ex2(x[j] - mmy[j]);
                lmy[j] += p[j];
            }
            // broadcast the weights of this row group's rows to all its lanes
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kVF; ++j) pbuf[rg * kV + ij[j]] = p[j];
            __syncwarp();
            float pv[kV];
            if constexpr (kV % 4 == 0) {
#pragma unroll
                for (int x4 = 0; x4 < kV; x4 += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(pbuf + rg * kV + x4);
                    pv[x4] = t.x, pv[x4 + 1] = t.y, pv[x4 + 2] = t.z, pv[x4 + 3] = t.w;
                }
            } else {
#pragma unroll
                for (int x1 = 0; x1 < kV; ++x1) pv[x1] = pbuf[rg * kV + x1];
            }
            // P.V into this lane's columns
#pragma unroll
            for (int rr = 0; rr < kRR; ++rr) {
                const int r = r0 + rr * kRW + rg;
#pragma unroll
                for (int nv = 0; nv < kNvec; ++nv) {
                    float f[kVec];
                    if constexpr (kFp8)
                        e4m3x8_to_f32(*reinterpret_cast<const uint2*>(vb + r * C::kKvRowBytes + (nv * kL + c) * 8), f);
                    else
                        E::to_f32(*reinterpret_cast<const uint4*>(vb + r * C::kKvRowBytes + (nv * kL + c) * 16), f);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float2 p2 = make_float2(pv[rr * G + h], pv[rr * G + h]);
#pragma unroll
                        for (int e = 0; e < kVec / 2; ++e)
                            acc[h][nv * kVec / 2 + e] =
                                __ffma2_rn(p2, make_float2(f[2 * e], f[2 * e + 1]), acc[h][nv * kVec / 2 + e]);
                    }
                }
            }
        }
        if (m.y & kSegEnd) finalize(m);
    };

    // ---- pipeline
    // a.test_extra_tx (test-only, normally 0): warp 0's first stage expects
    // bytes that never arrive, so that its bounded wait runs out.
#pragma unroll 1
    for (int s = 0; s < kStages; ++s) produce(s, (s == 0 && gwarp == 0) ? uint32_t(a.test_extra_tx) : 0u);
#pragma unroll 1
    for (int it = 0;; ++it) {
        const int slot = it % kStages;
        const uint32_t parity = uint32_t(it / kStages) & 1u;
        if (!mbar_wait_bounded(bar0 + 8 * slot, parity)) {
            if (lane == 0) atomicOr(a.flags, kFlagTimeout);
            // Let the copies already issued into the other stages land before leaving.
            for (int s = 1; s < kStages; ++s) {
                const int it2 = it + s;
                mbar_wait_bounded(bar0 + 8 * (it2 % kStages), uint32_t(it2 / kStages) & 1u);
            }
            break;
        }
        const int4 m = meta[slot];
        if (m.y & kEndOfWork) break;
        consume(slot, m);
        __syncwarp();
        produce(slot, 0u);
    }
    tails_finished(a, nwarps, lane);
}


}  // namespace pd
