// Batched decode attention over a paged (or contiguous) KV cache: the decode
// kernel and the kernel that merges its split results.
//
// Work decomposition. One "position" is one (kv head, head tile, listed page)
// triple; a pass over all listed pages is made for every (kv head, head tile).
// All positions of the call, total_pos = head_tiles * num_kv_heads * n_pos,
// are cut into equal contiguous ranges, one per warp of a grid sized to fill
// every SM. A warp therefore streams ~total_pos/warps pages regardless of how
// the lengths are spread over requests: a long request is split over several
// warps (split-KV), many short ones share a warp. Where a warp's range covers
// a request's whole page list the warp writes o and lse itself; otherwise it
// writes a normalised partial (o, lse) into the workspace slot (warp + segment),
// and merge_partials_kernel combines the partials in warp order.
//
// Inside a warp. The warp runs its own kStages-deep ring in shared memory.
// Lane 0 issues 1-D bulk async copies (cp.async.bulk) of whole K and V page
// slices -- in the HND layout rows [r0, r1) of one (page, kv head) are one
// contiguous block -- plus, at the start of a request, the group's q rows.
// Completion is counted in bytes on the stage's mbarrier. While stage s is
// being consumed, the next stages are in flight.
//
// Arithmetic (CUDA cores, f32). Lane (row group rg, column c) holds EPL
// elements of the head dimension for every q head of the group. For a round
// of RR rows it forms the group's partial dot products for those rows, then a
// reduce-scatter over the L lanes of the row group leaves each lane with a
// few complete scores. Softmax runs in log2 units (q is pre-scaled by
// sm_scale*log2 e) against a per-head reference maximum m that only moves
// when a score exceeds it by more than kTau; a move rescales the
// accumulators. P is broadcast through shared memory and every lane adds
// p * v into its accumulators for its columns. K and V bytes are read from
// HBM once for the whole group.
#pragma once

#include "pd_device.cuh"

namespace pd {

constexpr int kStages = 3;
constexpr int kChunkBytes = 4096;  // K bytes of one stage (V the same)
constexpr int kTableMax = 512;     // requests whose indptr / last_page_len are staged in smem
constexpr float kTau = 8.0f;       // reference max slack, log2 units: p <= 2^kTau

// Chunk metadata flags.
constexpr int kSegStart = 1, kSegEnd = 2, kSegComplete = 4, kEndOfWork = 8;

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

inline constexpr int table_bytes_for(bool staged) {
    return staged ? round_up((2 * kTableMax + 1) * 4, 128) : 0;
}

template <typename T, int D, int G>
struct Cfg {
    static constexpr int kEsz = int(sizeof(T));
    static constexpr int kVec = 16 / kEsz;           // elements per 16-byte vector
    static constexpr int kEpl = (G <= 4) ? 16 : 8;   // elements per lane per row
    static constexpr int kNvec = kEpl / kVec;        // vectors per lane per row
    static constexpr int kL = D / kEpl;              // lanes per row
    static constexpr int kRW = 32 / kL;              // rows side by side in a warp
    static constexpr int kRowBytes = D * kEsz;
    static constexpr int kRC = kChunkBytes / kRowBytes;  // rows per stage
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

template <typename T, int D, int G>
__global__ void __launch_bounds__(256, 1) decode_kernel(const DecodeArgs a) {
    using C = Cfg<T, D, G>;
    using E = Elt<T>;
    constexpr int kL = C::kL, kRW = C::kRW, kRR = C::kRR, kV = C::kV, kVF = C::kVF;
    constexpr int kVec = C::kVec, kNvec = C::kNvec, kEpl = C::kEpl, kRC = C::kRC;
    const float kNegInf = -__int_as_float(0x7f800000);

    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const bool contiguous = a.contiguous != 0;
    const bool staged = a.table_bytes > 0;
    int* s_indptr = reinterpret_cast<int*>(smem);
    int* s_lpl = s_indptr + kTableMax + 1;
    uint8_t* wsm = smem + a.table_bytes + wid * C::kWarpBytes;
    int4* meta = reinterpret_cast<int4*>(wsm + C::kMetaOff);
    const uint32_t bar0 = smem_u32(wsm + C::kBarOff);
    float* pbuf = reinterpret_cast<float*>(wsm + C::kPbufOff);

    // ---- set-up: stage the page table, zero the ring, init the barriers
    if (staged) {
        for (int x = threadIdx.x; x <= a.batch; x += blockDim.x) s_indptr[x] = __ldg(a.indptr + x);
        for (int x = threadIdx.x; x < a.batch; x += blockDim.x) s_lpl[x] = __ldg(a.last_page_len + x);
    }
    // Rows of a stage that no copy fills must still hold finite numbers, since
    // their (zero) softmax weight multiplies them.
    for (int off = lane * 16; off < kStages * C::kStageBytes; off += 32 * 16)
        *reinterpret_cast<uint4*>(wsm + off) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();  // the only block-wide barrier: warps are independent from here on

    const long long gwarp = (long long)blockIdx.x * nwarps + wid;
    const long long p0 = gwarp * a.pos_per_warp;
    const long long pend = min(p0 + a.pos_per_warp, a.total_pos);
    if (p0 >= pend) {
        launch_dependents();
        return;
    }

    const int B = a.batch, N = a.n_pos, P = a.page_size, Hk = a.num_kv_heads;
    const int HT = a.head_tiles, GT = a.heads_per_tile;
    auto indptr_at = [&](int b) -> int { return staged ? s_indptr[b] : __ldg(a.indptr + b); };
    auto range_of = [&](int b, int* lo, int* hi) {
        if (contiguous)
            request_range(b, N, true, a.npv, 0, 0, lo, hi);
        else
            request_range(b, N, false, 0, indptr_at(b), indptr_at(b + 1), lo, hi);
    };
    auto last_len = [&](int b) -> int {
        if (contiguous) return a.valid_kv_len - (a.npv - 1) * a.vpage;
        int v = staged ? s_lpl[b] : __ldg(a.last_page_len + b);
        if (v < 0 || v > P) {
            if (lane == 0) atomicOr(a.flags, kFlagBadLastPageLen);
            v = v < 0 ? 0 : P;
        }
        return v;
    };
    // First request whose range ends after position i (B if none).
    auto find_request = [&](int i) -> int {
        if (contiguous) return min(i / a.npv, B);
        int lo = 0, hi = B;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (indptr_at(mid + 1) > i) hi = mid;
            else lo = mid + 1;
        }
        return lo;
    };

    // ---- producer walk state (identical in every lane)
    long long wp = p0;  // next position to emit
    int wsh = int(p0 / N), wi = int(p0 % N);
    int wb = find_request(wi), wlo = 0, whi = 0, wj = 0;
    if (wb < B) range_of(wb, &wlo, &whi);
    bool wfirst = true;
    // Window of 64 page ids: win0 = indices[wbase + lane], win1 = indices[wbase + 32 + lane].
    int wbase = -64, win0 = -1, win1 = -1;
    auto idx_load = [&](int x) -> int { return (x >= 0 && x < N) ? __ldg(a.indices + x) : -1; };
    auto page_id = [&](int i) -> int {
        if (i < wbase || i >= wbase + 64) {
            wbase = i & ~31;
            win0 = idx_load(wbase + lane);
            win1 = idx_load(wbase + 32 + lane);
        } else if (i >= wbase + 32) {
            wbase += 32;
            win0 = win1;
            win1 = idx_load(wbase + 32 + lane);
        }
        return __shfl_sync(kFull, win0, i - wbase);
    };
    const uint64_t policy = l2_evict_first_policy();
    const size_t row_bytes = size_t(C::kRowBytes);

    // Emit the next chunk into `slot` (whole warp; lane 0 issues the copies).
    auto produce = [&](int slot) {
        while (wp < pend) {
            if (wb >= B) {  // past the last request of this pass: next pass
                wp += N - wi;
                ++wsh;
                wi = 0;
                wj = 0;
                wb = find_request(0);
                if (wb < B) range_of(wb, &wlo, &whi);
                continue;
            }
            if (wi >= whi) {
                ++wb;
                if (wb < B) range_of(wb, &wlo, &whi);
                continue;
            }
            if (wi < wlo) {  // positions before this request belong to none
                wp += wlo - wi;
                wi = wlo;
                wj = 0;
                continue;
            }
            break;
        }
        const uint32_t bar = bar0 + 8 * slot;
        uint8_t* st = wsm + slot * C::kStageBytes;
        if (wp >= pend) {
            if (lane == 0) {
                meta[slot] = make_int4(0, kEndOfWork, 0, 0);
                mbar_arrive(bar);
            }
            return;
        }
        const int kh = wsh / HT, ht = wsh % HT;
        int valid, page;
        size_t src_row;  // element row index of the page slice's row 0
        if (contiguous) {
            page = wi - wlo;
            valid = (wi == whi - 1) ? last_len(wb) : a.vpage;
            src_row = (size_t(wb) * Hk + kh) * size_t(a.max_kv_len) + size_t(page) * a.vpage;
        } else {
            page = page_id(wi);
            valid = (wi == whi - 1) ? last_len(wb) : P;
            if (page < 0 || page >= a.num_total_pages) {
                if (lane == 0) atomicOr(a.flags, kFlagBadPage);
                valid = 0;
                page = 0;
            }
            src_row = (size_t(page) * Hk + kh) * size_t(P);
        }
        const int nck = valid > kRC ? (valid + kRC - 1) / kRC : 1;
        int rows = valid - wj * kRC;
        rows = rows < 0 ? 0 : (rows > kRC ? kRC : rows);
        int flags = 0;
        if (wfirst || (wi == wlo && wj == 0)) flags |= kSegStart;
        if (wj == nck - 1 && (wi == whi - 1 || wp + 1 == pend)) flags |= kSegEnd;
        const long long seg_lo = (long long)wsh * N + wlo, seg_hi = (long long)wsh * N + whi;
        if (seg_lo >= p0 && seg_hi <= pend) flags |= kSegComplete;
        if (lane == 0) {
            meta[slot] = make_int4(rows, flags, wb, wsh);
            const uint32_t kv_bytes = uint32_t(rows) * uint32_t(row_bytes);
            const uint32_t q_bytes = (flags & kSegStart) ? uint32_t(GT * C::kRowBytes) : 0u;
            const uint32_t total = 2 * kv_bytes + q_bytes;
            if (total == 0) {
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, total);
                if (kv_bytes) {
                    const size_t off = (src_row + size_t(wj) * kRC) * row_bytes;
                    bulk_g2s(smem_u32(st), static_cast<const uint8_t*>(a.k) + off, kv_bytes, bar, policy);
                    bulk_g2s(smem_u32(st + kChunkBytes), static_cast<const uint8_t*>(a.v) + off, kv_bytes,
                             bar, policy);
                }
                if (q_bytes) {
                    const size_t qoff = (size_t(wb) * a.num_qo_heads + size_t(kh) * a.group +
                                         size_t(ht) * GT) * row_bytes;
                    bulk_g2s(smem_u32(st + 2 * kChunkBytes), static_cast<const uint8_t*>(a.q) + qoff, q_bytes,
                             bar);
                }
            }
        }
        wfirst = false;
        if (++wj == nck) {
            wj = 0;
            ++wp;
            if (++wi == N) {
                ++wsh;
                wi = 0;
                wb = find_request(0);
                if (wb < B) range_of(wb, &wlo, &whi);
            }
        }
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

    float qf[G][kEpl];
    float acc[G][kEpl];
    float mref[G];
    float mmy[kVF], lmy[kVF];
    auto reset_state = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mref[h] = kNegInf;
#pragma unroll
            for (int e = 0; e < kEpl; ++e) acc[h][e] = 0.f;
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

    auto finalize = [&](int4 m) {
        float lh[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kVF; ++j) s += (primary && hj[j] == h) ? lmy[j] : 0.f;
            lh[h] = warp_sum(s);
        }
#pragma unroll
        for (int off = kL; off < 32; off <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < kEpl; ++e) acc[h][e] += __shfl_xor_sync(kFull, acc[h][e], off);
        const int b = m.z, sh = m.w;
        const int kh = sh / HT, ht = sh % HT;
        const int head0 = kh * a.group + ht * GT;
        if (m.y & kSegComplete) {
            if (lane < kL) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (h >= GT) break;
                    const float inv = lh[h] > 0.f ? 1.0f / lh[h] : 0.f;
                    T* orow = static_cast<T*>(a.o) + (size_t(b) * a.num_qo_heads + head0 + h) * D;
#pragma unroll
                    for (int nv = 0; nv < kNvec; ++nv) {
                        float f[kVec];
#pragma unroll
                        for (int e = 0; e < kVec; ++e) f[e] = acc[h][nv * kVec + e] * inv;
                        *reinterpret_cast<uint4*>(orow + (nv * kL + c) * kVec) = E::from_f32(f);
                    }
                }
            }
            if (a.lse != nullptr && lane < GT) {
                const float l = pick(lh, lane), mr = pick(mref, lane);
                a.lse[size_t(b) * a.num_qo_heads + head0 + lane] = l > 0.f ? (mr + log2f(l)) * kLn2 : kNegInf;
            }
        } else {
            const long long slot = gwarp + (long long)sh * B + b;
            if (lane < kL) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    if (h >= GT) break;
                    const float inv = lh[h] > 0.f ? 1.0f / lh[h] : 0.f;
                    float* prow = a.part_o + (size_t(slot) * G + h) * D;
#pragma unroll
                    for (int nv = 0; nv < kNvec; ++nv)
#pragma unroll
                        for (int e4 = 0; e4 < kVec; e4 += 4)
                            *reinterpret_cast<float4*>(prow + (nv * kL + c) * kVec + e4) =
                                make_float4(acc[h][nv * kVec + e4] * inv, acc[h][nv * kVec + e4 + 1] * inv,
                                            acc[h][nv * kVec + e4 + 2] * inv, acc[h][nv * kVec + e4 + 3] * inv);
                }
            }
            if (lane < GT) {
                const float l = pick(lh, lane), mr = pick(mref, lane);
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
                    for (int e = 0; e < kVec; ++e) qf[h][nv * kVec + e] = f[e] * a.q_scale;
                }
        }
        const int rows = m.x;
#pragma unroll
        for (int rd = 0; rd < C::kRounds; ++rd) {
            const int r0 = rd * kRW * kRR;
            if (r0 >= rows) break;
            // scores: partial dot products of this lane's columns
            float part[kV];
#pragma unroll
            for (int x = 0; x < kV; ++x) part[x] = 0.f;
#pragma unroll
            for (int rr = 0; rr < kRR; ++rr) {
                const int r = r0 + rr * kRW + rg;
#pragma unroll
                for (int nv = 0; nv < kNvec; ++nv) {
                    float f[kVec];
                    E::to_f32(*reinterpret_cast<const uint4*>(kb + r * C::kRowBytes + (nv * kL + c) * 16), f);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < kVec; ++e)
                            part[rr * G + h] = fmaf(qf[h][nv * kVec + e], f[e], part[rr * G + h]);
                }
            }
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
#pragma unroll
                    for (int e = 0; e < kEpl; ++e) acc[h][e] *= alpha[h];
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
                    E::to_f32(*reinterpret_cast<const uint4*>(vb + r * C::kRowBytes + (nv * kL + c) * 16), f);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < kVec; ++e)
                            acc[h][nv * kVec + e] = fmaf(pv[rr * G + h], f[e], acc[h][nv * kVec + e]);
                }
            }
        }
        if (m.y & kSegEnd) finalize(m);
    };

    // ---- pipeline
#pragma unroll 1
    for (int s = 0; s < kStages; ++s) produce(s);
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
        produce(slot);
    }
    launch_dependents();
}

// One warp per (request, kv head, head tile, q head): combine the partial
// results the decode warps wrote for a request split across warps, in warp
// order; write zeros / -inf for requests with no pages.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_partials_kernel(const MergeArgs a) {
    constexpr int kPer = D / 32;  // elements per lane
    const float kNegInf = -__int_as_float(0x7f800000);
    grid_dependency_wait();  // the decode kernel's partials are complete and visible
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
    if (hi > lo) {
        const long long first = ((long long)sh * a.n_pos + lo) / a.pos_per_warp;
        const long long last = ((long long)sh * a.n_pos + hi - 1) / a.pos_per_warp;
        if (first == last) return;  // one warp held the whole request and wrote it
        const int parts = int(last - first + 1);
        auto slot_of = [&](int cpart) { return (first + cpart + s) * a.G + h; };
        float M = kNegInf;
        for (int cp = lane; cp < parts; cp += 32) M = fmaxf(M, a.part_lse[slot_of(cp)]);
        M = warp_max(M);
        if (M != kNegInf) {
            float S = 0.f;
            for (int cp = lane; cp < parts; cp += 32) S += ex2(a.part_lse[slot_of(cp)] - M);
            S = warp_sum(S);
            L = M + log2f(S);
            for (int cp = 0; cp < parts; ++cp) {
                const long long sl = slot_of(cp);
                const float w = ex2(a.part_lse[sl] - L);
                const float* po = a.part_o + size_t(sl) * D + lane * kPer;
#pragma unroll
                for (int e = 0; e < kPer; e += 2) {
                    const float2 t = *reinterpret_cast<const float2*>(po + e);
                    acc[e] = fmaf(w, t.x, acc[e]);
                    acc[e + 1] = fmaf(w, t.y, acc[e + 1]);
                }
            }
        }
    }
    // Each lane writes its kPer consecutive elements.
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<float2*>(reinterpret_cast<float*>(orow) + lane * kPer + e) = make_float2(acc[e], acc[e + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < kPer; e += 2) {
            const uint32_t w = Elt<T>::pack(acc[e], acc[e + 1]);
            *reinterpret_cast<uint32_t*>(orow + lane * kPer + e) = w;
        }
    }
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
    auto lse2 = [&](int cp) { return lse_parts[size_t(cp) * num_rows + row] * kLog2e; };
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    float M = kNegInf;
    for (int cp = lane; cp < num_parts; cp += 32) M = fmaxf(M, lse2(cp));
    M = warp_max(M);
    float L = kNegInf;
    if (M != kNegInf) {
        float S = 0.f;
        for (int cp = lane; cp < num_parts; cp += 32) S += ex2(lse2(cp) - M);
        S = warp_sum(S);
        L = M + log2f(S);
        for (int cp = 0; cp < num_parts; ++cp) {
            const float w = ex2(lse2(cp) - L);
            const float* po = o_parts + (size_t(cp) * num_rows + row) * D + lane * kPer;
#pragma unroll
            for (int e = 0; e < kPer; e += 2) {
                const float2 t = *reinterpret_cast<const float2*>(po + e);
                acc[e] = fmaf(w, t.x, acc[e]);
                acc[e + 1] = fmaf(w, t.y, acc[e + 1]);
            }
        }
    }
    T* orow = static_cast<T*>(o) + size_t(row) * D;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<float2*>(reinterpret_cast<float*>(orow) + lane * kPer + e) = make_float2(acc[e], acc[e + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < kPer; e += 2)
            *reinterpret_cast<uint32_t*>(orow + lane * kPer + e) = Elt<T>::pack(acc[e], acc[e + 1]);
    }
    if (lse && lane == 0) lse[row] = (L == kNegInf) ? kNegInf : L * kLn2;
}

// Kernels and sizes for one (T, D, G) combination, handed to the host code.
struct KernelSet {
    const void* decode;
    const void* merge;
    const void* merge_states;
    int warp_bytes;      // dynamic shared memory per decode warp
    int rows_per_stage;  // K (and V) rows one pipeline stage holds
};

template <typename T>
bool lookup_kernels_t(int D, int G, KernelSet* ks) {
#define PD_CASE(DD, GG)                                                        \
    if (D == DD && G == GG) {                                                  \
        ks->decode = reinterpret_cast<const void*>(decode_kernel<T, DD, GG>);  \
        ks->merge = reinterpret_cast<const void*>(merge_partials_kernel<T, DD>); \
        ks->merge_states = reinterpret_cast<const void*>(merge_states_kernel<T, DD>); \
        ks->warp_bytes = Cfg<T, DD, GG>::kWarpBytes;                           \
        ks->rows_per_stage = Cfg<T, DD, GG>::kRC;                              \
        return true;                                                           \
    }
    PD_CASE(64, 1) PD_CASE(64, 2) PD_CASE(64, 4) PD_CASE(64, 8)
    PD_CASE(128, 1) PD_CASE(128, 2) PD_CASE(128, 4) PD_CASE(128, 8)
    PD_CASE(256, 1) PD_CASE(256, 2) PD_CASE(256, 4) PD_CASE(256, 8)
#undef PD_CASE
    return false;
}

}  // namespace pd
