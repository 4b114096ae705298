// Batched decode attention over E4M3 (FP8) paged pools on tensor cores, for
// tiles of 4..8 q heads per kv head at head_dim 128 / 256. Element value =
// E4M3 code value * scale[kv head] (k_scale for K, v_scale for V).
//
// An E4M3 byte is a whole element, so per byte of HBM the arithmetic of the
// group doubles against a 16-bit pool: the CUDA cores cannot keep up, and a
// warp that moves one 16-row page per pipeline step spends more time on the
// step's fixed work (barrier wait, walk, softmax bookkeeping) than the page's
// bytes take to arrive. This kernel therefore:
//  - stages up to two pages of the same segment per pipeline slot at head_dim
//    128 (32 tokens, two independent 16-token score tiles). The codes come
//    through tensor maps in boxes of 16 rows x 128 bytes with the 128-byte
//    swizzle (16-byte piece x of row r lands at piece x ^ (r & 7)), which
//    keeps the reads below free of bank conflicts;
//  - builds the K operand of the score mma straight from the codes in shared
//    memory, widening them in registers (every E4M3 value is an f16 value, so
//    the f16 mma sees them exactly). The 16 dims of k step kk = 4j + t that
//    lane (g, c) holds are not the mma's canonical columns but dims
//    k_base(c, j) + 4t + {0..3}, k_base = 128 (j >> 1) + 32c + 16 (j & 1):
//    one 16-byte load per row feeds four k steps, and the 8 lanes of one
//    load phase read 8 different 16-byte pieces. q takes the same
//    permutation, so the dot products are unchanged. Score row g of a tile
//    holds token 2g - (g & 1) and row g + 8 that token + 2 (see below);
//  - builds the V operand of the P.V mma with the transposing 8-bit
//    ldmatrix (16 tokens x 16 dims per matrix): it hands lane (g, c) the
//    codes of tokens 4c .. 4c+3 of dims g and g + 8, which is the A
//    fragment of m tile "16 dims" once each token pair is widened, with the
//    mma's k index 2c, 2c+1 standing for tokens 4c, 4c+1 and 2c+8, 2c+9 for
//    4c+2, 4c+3. The score rows' token order above makes P leave movmatrix
//    in that same order. No shared-memory tile is written: a stage holds
//    only the copied codes;
//  - keeps q in f16 as q 2^-e, e a power of two per head that puts its
//    largest |q| into [2^14, 2^15): a bf16 or f16 q is then exact in f16 (an
//    element more than 2^28 below the largest keeps an error under 2^-24 of
//    it), one mma per k step forms the dot products, and 2^e, sm_scale,
//    log2 e and k_scale multiply the f32 sums. P enters in f16 alone (V is
//    exact in f16, so P's rounding costs o no more than its own f16
//    rounding). q is not staged with the pages:
//    the producer pulls a segment's q rows into L2 with its first stage, and
//    the consumer loads its fragments from there, which keeps a warp's shared
//    memory to its two stages of codes.
// Work partition, walk, softmax and the partial-result layout (8 heads per
// slot) are those of decode_mma_kernel.
#pragma once

#include <type_traits>

#include "pd_decode_mma.cuh"

namespace pd {

// Two 16 x 16 byte matrices from shared memory, transposed: lanes 0-15 give
// the addresses of matrix 0's rows, lanes 16-31 those of matrix 1. Lane
// 4 g + q receives rows 4q .. 4q+3 of byte column g (r[0]) and of column g + 8
// (r[1]) of matrix 0, and the same of matrix 1 in r[2], r[3].
__device__ __forceinline__ void ldsm_b8_x2_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <int D>
struct CfgF8 {
    // Two stages of two pages and up to 12 warps per block at head_dim 128
    // (registers and shared memory both stop there): measured faster than
    // 3 such stages x 8 warps, and than 3 one-page stages x 16 warps, whose
    // extra warps do not pay for twice the per-stage work per byte.
    // At 256 the registers of 12 warps would not hold the accumulators: 8.
    static constexpr int kStages = 2;
    static constexpr int kMaxWarps = D <= 128 ? 12 : 8;
    // 16-row tiles per stage: two at head_dim 128 (8 KB of K and V codes per
    // stage), one at 256 (a tile is 4 KB already).
    static constexpr int kSub = D <= 128 ? 2 : 1;
    static constexpr int kTileRaw = kMmaRows * D;      // E4M3 bytes of one K (or V) tile
    static constexpr int kBoxes = D / 128;             // 128-byte column boxes per tile
    static constexpr int kBoxBytes = kMmaRows * 128;   // one box: 16 rows x 128 codes

    static constexpr int kVOff = kSub * kTileRaw;      // V tiles within a stage
    // q is not staged: it is read at a segment start, from L2 (see produce)
    static constexpr int kStageBytes = round_up(2 * kSub * kTileRaw, 128);
    static constexpr int kMetaOff = kStages * kStageBytes;
    static constexpr int kBarOff = kMetaOff + kStages * 16;
    // stages stay 1024-byte aligned for the swizzle
    static constexpr int kWarpBytes = round_up(kBarOff + kStages * 8, 1024);
    static constexpr int kKSteps = D / 16;
    static constexpr int kJ = D / 64;  // 64-dim groups: one 16-byte load per row each
};

template <typename T, int D>
__global__ void __launch_bounds__(CfgF8<D>::kMaxWarps * 32, 1)
    decode_fp8_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv) {
    static_assert(D == 128 || D == 256, "head_dim 128 or 256");
    using C = CfgF8<D>;
    using M = __half;  // mma operand type
    constexpr int kS = C::kStages, kKS = C::kKSteps;
    constexpr float kShift = 7.f;  // f16 P: weights kept 2^7 larger, taken out of lse
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

    const long long gwarp = (long long)blockIdx.x * nwarps + wid;
    const long long p0 = gwarp * a.pos_per_warp;
    const long long pend = min(p0 + a.pos_per_warp, a.total_pos);
    Walk<false> walk(a, s_indptr, s_lpl, p0, pend, lane);
    const int first_page = walk.prefetch_first();
    const int GT = a.heads_per_tile;
    if (lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }

    walk.stage_table(s_indptr, s_lpl, [&] {
        if (lane == 0) {
            for (int s = 0; s < kS; ++s) mbar_init(bar0 + 8 * s, 1);
            fence_mbar_init();
        }
        // The first stage's positions: on the Llama-shaped batch, pulling in
        // 4, 8 or 12 positions measured slower, and none slower still.
        walk.template prefetch_first_slabs<false>(first_page, C::kSub, size_t(D));
    });
    __syncthreads();  // the only block-wide barrier
    launch_dependents();
    if (p0 >= pend) return;
    walk.build(p0, first_page);

    const uint64_t policy = l2_evict_first_policy();
    const size_t q_row_bytes = size_t(D) * sizeof(T);
    // Emit the next one or two chunks into `slot`. A chunk without kSegEnd
    // is always followed by one of the same segment (same request and kv
    // head): a second chunk is taken only then, so a stage never spans two
    // segments.
    auto produce = [&](int slot, uint32_t extra_tx) {
        Chunk c0, c1;
        const bool have = walk.template next<kMmaRows>(&c0);
        const bool two = (C::kSub == 2 && have && !(c0.flags & kSegEnd)) ? walk.template next<kMmaRows>(&c1) : false;
        if (lane != 0) return;
        const uint32_t bar = bar0 + 8 * slot;
        const uint32_t st = wsm_u32 + slot * C::kStageBytes;
        if (!have) {
            meta[slot] = make_int4(0, kEndOfWork, 0, 0);
            mbar_arrive(bar);
            return;
        }
        const int r1 = two ? c1.rows : 0;
        const int flags = two ? ((c0.flags & ~kSegEnd) | (c1.flags & kSegEnd)) : c0.flags;
        meta[slot] = make_int4(c0.rows | (r1 << 16), flags, c0.qrow, c0.seg);
        // A segment's q rows are pulled into L2 with its first stage; the
        // consumer reads them from there when it reaches that stage.
        if (flags & kSegStart)
            bulk_prefetch_l2(static_cast<const uint8_t*>(a.q) + size_t(c0.qrow) * q_row_bytes,
                             uint32_t(GT * q_row_bytes));
        // A tile with rows lands as whole boxes (rows outside the page read as zero).
        const int n0 = c0.rows > 0, n1 = r1 > 0;
        const uint32_t total = uint32_t(n0 + n1) * 2u * uint32_t(C::kTileRaw);
        if (total == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, total + extra_tx);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
            if (n0) {
                tma_load_4d(st + bx * C::kBoxBytes, &tmk, bx * 128, c0.row0, c0.kh, c0.slab, bar, policy);
                tma_load_4d(st + C::kVOff + bx * C::kBoxBytes, &tmv, bx * 128, c0.row0, c0.kh, c0.slab, bar, policy);
            }
            if (n1) {
                tma_load_4d(st + C::kTileRaw + bx * C::kBoxBytes, &tmk, bx * 128, c1.row0, c1.kh, c1.slab, bar,
                            policy);
                tma_load_4d(st + C::kVOff + C::kTileRaw + bx * C::kBoxBytes, &tmv, bx * 128, c1.row0, c1.kh,
                            c1.slab, bar, policy);
            }
        }
    };

    // ---- consumer state: lane (g, c) owns tokens g, g+8 of each tile and heads 2c, 2c+1
    const int g = lane >> 2, c = lane & 3;
    uint32_t qh[kKS][2];  // score-mma B fragments (permuted dims): q 2^-e in f16, exact
    float qsc0 = 0.f, qsc1 = 0.f;  // 2^e * sm_scale * log2 e * k_scale of heads 2c and 2c + 1
    float acc[kKS][4];  // P.V accumulators: o^T[v_dim(mt, 0 / 1)][head 2c (+1)]
    // The dim that accumulator row g (hi = 0) or g + 8 (hi = 1) of m tile mt stands for.
    auto v_dim = [&](int mt, int hi) { return 16 * mt + 8 * hi + g; };
    // Score row g of a tile holds token rg0 and row g + 8 token rg0 + 2, so
    // that P leaves movmatrix with lane (g, c) holding tokens 4c .. 4c+3: the
    // order in which ldmatrix hands out the V codes.
    const int rg0 = 2 * g - (g & 1);
    float m0, m1, l0, l1;
    auto reset_state = [&]() {
#pragma unroll
        for (int mt = 0; mt < kKS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        m0 = m1 = kNegInf;
        l0 = l1 = 0.f;
    };
    reset_state();
#pragma unroll
    for (int kk = 0; kk < kKS; ++kk) qh[kk][0] = qh[kk][1] = 0u;

    auto finalize = [&](int4 m) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        const int qrow = m.z;
        const int h0 = 2 * c, h1 = 2 * c + 1;
        const float vsc = __ldg(a.v_scale + (qrow % a.num_qo_heads) / a.group);  // V scale, applied once
        const float inv0 = l0 > 0.f ? vsc / l0 : 0.f, inv1 = l1 > 0.f ? vsc / l1 : 0.f;
        const float lse0 = l0 > 0.f ? m0 - kShift + log2f(l0) : kNegInf;
        const float lse1 = l1 > 0.f ? m1 - kShift + log2f(l1) : kNegInf;
        if (m.y & kSegComplete) {
            T* o0 = static_cast<T*>(a.o) + (size_t(qrow) + h0) * D;
            T* o1 = o0 + D;
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                const int d = v_dim(mt, 0), d8 = v_dim(mt, 1);
                if (h0 < GT) {
                    o0[d] = T(acc[mt][0] * inv0);
                    o0[d8] = T(acc[mt][2] * inv0);
                }
                if (h1 < GT) {
                    o1[d] = T(acc[mt][1] * inv1);
                    o1[d8] = T(acc[mt][3] * inv1);
                }
            }
            if (g == 0 && a.lse != nullptr) {
                if (h0 < GT) a.lse[size_t(qrow) + h0] = lse0 == kNegInf ? kNegInf : lse0 * kLn2;
                if (h1 < GT) a.lse[size_t(qrow) + h1] = lse1 == kNegInf ? kNegInf : lse1 * kLn2;
            }
        } else {
            const long long slot = gwarp + m.w;
            float* p0r = a.part_o + (size_t(slot) * 8 + h0) * D;
            float* p1r = p0r + D;
#pragma unroll
            for (int mt = 0; mt < kKS; ++mt) {
                const int d = v_dim(mt, 0), d8 = v_dim(mt, 1);
                if (h0 < GT) {
                    p0r[d] = acc[mt][0] * inv0;
                    p0r[d8] = acc[mt][2] * inv0;
                }
                if (h1 < GT) {
                    p1r[d] = acc[mt][1] * inv1;
                    p1r[d8] = acc[mt][3] * inv1;
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
        const uint8_t* stp = wsm + slot * C::kStageBytes;
        const int rows[2] = {m.x & 0xffff, m.x >> 16};
        if (m.y & kSegStart) {
            // q of head g at the permuted dims of k step kk = 4j + t:
            // k_base(c, j) + 4t + {0, 1} (first register), + {2, 3} (second),
            // scaled by a power of two 2^-e (the head's largest |q| into
            // [2^14, 2^15)): a bf16 or f16 q is then exact in f16, and 2^e and
            // the scales multiply the f32 sums.
            const float qs = a.q_scale * __ldg(a.k_scale + (m.z % a.num_qo_heads) / a.group);
            const uint8_t* qb = static_cast<const uint8_t*>(a.q) + (size_t(m.z) + g) * q_row_bytes;
            uint2 w[kKS];
            float mx = 0.f;
#pragma unroll
            for (int kk = 0; kk < kKS; ++kk) {
                const int j = kk >> 2;
                const int d0 = 128 * (j >> 1) + 32 * c + 16 * (j & 1) + 4 * (kk & 3);
                w[kk] = make_uint2(0u, 0u);
                if (g < GT) w[kk] = __ldg(reinterpret_cast<const uint2*>(qb + d0 * 2));
                const float2 v0 = unpack_pair<T>(w[kk].x), v1 = unpack_pair<T>(w[kk].y);
                mx = fmaxf(fmaxf(mx, fmaxf(fabsf(v0.x), fabsf(v0.y))), fmaxf(fabsf(v1.x), fabsf(v1.y)));
            }
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            const int e = mx > 0.f ? max(-100, min(100, ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14)) : 0;
            const float inv = __int_as_float((127 - e) << 23);
#pragma unroll
            for (int kk = 0; kk < kKS; ++kk) {
                const float2 v0 = unpack_pair<T>(w[kk].x), v1 = unpack_pair<T>(w[kk].y);
                qh[kk][0] = pack_pair<M>(v0.x * inv, v0.y * inv);
                qh[kk][1] = pack_pair<M>(v1.x * inv, v1.y * inv);
            }
            // the scales of heads 2c and 2c + 1, from lanes 8c (g = 2c) and 8c + 4
            const int e0 = __shfl_sync(kFull, e, 8 * c), e1 = __shfl_sync(kFull, e, 8 * c + 4);
            qsc0 = qs * __int_as_float((127 + e0) << 23);
            qsc1 = qs * __int_as_float((127 + e1) << 23);
        }
        // scores of both tiles: S_s[16 tokens][8 heads], K fragments from the
        // codes; the k steps of both tiles interleave: two independent mma chains.
        float sc[2][4];
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[s][i] = 0.f;
#pragma unroll
        for (int j = 0; j < C::kJ; ++j) {
            uint32_t xa[2][4], xb[2][4];
#pragma unroll
            for (int s = 0; s < C::kSub; ++s) {
                // token rows rg0 and rg0 + 2 of the box holding this 16-byte piece (2c + (j & 1))
                const uint8_t* kb = stp + s * C::kTileRaw + (j >> 1) * C::kBoxBytes;
                const int pc = 2 * c + (j & 1);
                const uint4 wa = *reinterpret_cast<const uint4*>(kb + rg0 * 128 + ((pc ^ (rg0 & 7)) << 4));
                const uint4 wb =
                    *reinterpret_cast<const uint4*>(kb + (rg0 + 2) * 128 + ((pc ^ ((rg0 + 2) & 7)) << 4));
                xa[s][0] = wa.x, xa[s][1] = wa.y, xa[s][2] = wa.z, xa[s][3] = wa.w;
                xb[s][0] = wb.x, xb[s][1] = wb.y, xb[s][2] = wb.z, xb[s][3] = wb.w;
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int kk = 4 * j + t;
#pragma unroll
                for (int s = 0; s < C::kSub; ++s) {
                    if (rows[s] == 0) continue;
                    const uint32_t af[4] = {e4m3x2_to_f16x2(xa[s][t]), e4m3x2_to_f16x2(xb[s][t]),
                                            e4m3x2_to_f16x2(xa[s][t] >> 16), e4m3x2_to_f16x2(xb[s][t] >> 16)};
                    mma_16816<M>(sc[s], af, qh[kk][0], qh[kk][1]);
                }
            }
        }
        // softmax over the 32 tokens; x[s][i]: tile s, token g (i = 0, 1) or
        // g + 8 (i = 2, 3), head 2c (i even) or 2c + 1 (i odd)
        float x[2][4];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            x[s][0] = rg0 < rows[s] ? sc[s][0] * qsc0 : kNegInf;
            x[s][1] = rg0 < rows[s] ? sc[s][1] * qsc1 : kNegInf;
            x[s][2] = rg0 + 2 < rows[s] ? sc[s][2] * qsc0 : kNegInf;
            x[s][3] = rg0 + 2 < rows[s] ? sc[s][3] * qsc1 : kNegInf;
        }
        const float c0l = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
        const float c1l = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
        if (__any_sync(kFull, c0l > m0 + kTauM || c1l > m1 + kTauM)) {
            float c0 = c0l, c1 = c1l;
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
        // P.V B fragments of each tile: P in f16 alone. V is exact in f16, so
        // P's rounding (2^-11 of each weight) moves o by at most 2^-11 max|v|,
        // the order of o's own f16 rounding; l sums the unrounded weights.
        uint32_t bh[2][2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const float p0 = x[s][0] == kNegInf ? 0.f : ex2(x[s][0] - m0 + kShift);
            const float p1 = x[s][1] == kNegInf ? 0.f : ex2(x[s][1] - m1 + kShift);
            const float p2 = x[s][2] == kNegInf ? 0.f : ex2(x[s][2] - m0 + kShift);
            const float p3 = x[s][3] == kNegInf ? 0.f : ex2(x[s][3] - m1 + kShift);
            l0 += p0 + p2;
            l1 += p1 + p3;
            bh[s][0] = movm_trans(pack_pair<M>(p0, p1));
            bh[s][1] = movm_trans(pack_pair<M>(p2, p3));
        }
        // O^T[head_dim][8 heads] += V_s^T[head_dim][16 tokens] P_s[16 tokens][8 heads]. m tile mt
        // holds dims 16 mt .. 16 mt + 15; ldmatrix hands lane (g, c) the codes of tokens
        // 4c .. 4c+3 of dims g and g + 8, which is the A fragment once the token pairs
        // are widened (k index 2c, 2c+1 <-> tokens 4c, 4c+1; 2c+8, 2c+9 <-> 4c+2, 4c+3).
        // Tokens past the valid length are zeroed, so that their zero weights never
        // meet a NaN code.
        const int tr = lane & 15;  // the token row whose address this lane gives
#pragma unroll
        for (int s = 0; s < C::kSub; ++s) {
            if (rows[s] == 0) continue;
            const int rv = rows[s] - 4 * c;
            const uint32_t vmask = rv >= 4 ? 0xffffffffu : rv <= 0 ? 0u : (0xffffffffu >> (8 * (4 - rv)));
            const uint32_t vt = wsm_u32 + uint32_t(slot * C::kStageBytes + C::kVOff + s * C::kTileRaw);
#pragma unroll
            for (int mp = 0; mp < kKS / 2; ++mp) {
                const int mt0 = 2 * mp + (lane >> 4);  // the m tile of this lane's row address
                const uint32_t addr =
                    vt + uint32_t((mt0 >> 3) * C::kBoxBytes + tr * 128 + (((mt0 & 7) ^ (tr & 7)) << 4));
                uint32_t r[4];
                ldsm_b8_x2_trans(addr, r);
                if (rows[s] < kMmaRows) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) r[i] &= vmask;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t af[4] = {e4m3x2_to_f16x2(r[2 * h]), e4m3x2_to_f16x2(r[2 * h + 1]),
                                            e4m3x2_to_f16x2(r[2 * h] >> 16), e4m3x2_to_f16x2(r[2 * h + 1] >> 16)};
                    mma_16816<M>(acc[2 * mp + h], af, bh[s][0], bh[s][1]);
                }
            }
        }
        if (m.y & kSegEnd) finalize(m);
    };

    // a.test_extra_tx (test-only, normally 0): warp 0's first stage expects
    // bytes that never arrive, so that its bounded wait runs out.
#pragma unroll 1
    for (int s = 0; s < kS; ++s) produce(s, (s == 0 && gwarp == 0) ? uint32_t(a.test_extra_tx) : 0u);
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
        produce(slot, 0u);
    }
}

}  // namespace pd
