// Batched decode attention over E4M3 (FP8) paged pools on the 5th-generation
// tensor cores (tcgen05.mma kind::f8f6f4, accumulators in tensor memory), for
// groups of 4 q heads per kv head at head_dim 128 with bf16 q and o and an
// even number of kv heads. Element value = E4M3 code value * scale[kv head]
// (k_scale for K, v_scale for V).
//
// An E4M3 byte is a whole element, so the arithmetic per byte of HBM doubles
// against a 16-bit pool. mma.sync takes 16-bit operands only (its E4M3 form is
// carried out as f16 mma after widening), so a warp-level kernel has to widen
// every code in registers and runs out of issue slots before it runs out of
// bandwidth. Here the tensor cores read the codes where the copies put them.
//
// Partition: the kv heads are taken in pairs, each pair with its 8 q heads as
// one head tile (the host presents the pair as one kv head of group 8, so the
// walk, the partial slots and the merge are those of decode_mma_kernel), and
// positions (pair, page) are cut into equal shares. A share streams in tiles
// of up to 4 pages of one segment (request, pair): 4 x 2 x 16 = 128 K/V rows,
// one tensor-map box of 16 rows x 2 kv heads (4 KB) per page for K and for V.
//
// Roles: two independent pipelines per block (tensor memory holds a kernel to
// one block per SM), pipeline p with a share, shared memory, tensor-memory
// columns and barriers of its own, and 6 warps:
//  - warp 8 + p, producer: walks the share; per tile issues the copies into a
//    3-stage ring (128-byte swizzle, so that the 128 rows of a tile form one
//    operand in the canonical swizzled layout), and writes beside them the
//    tile's metadata and the E4M3 parts of its 8 q rows;
//  - warp 10 + p, lane 0, mma: S[128 rows][16] = K q^T (A = K, K-major; B =
//    the q parts, K-major; 4 k steps of 32 dims), and, once the softmax warps
//    have written P, O^T[128 dims][16] = V^T P (A = V read MN-major from the
//    same tile; B = the P parts, K-major; 4 k steps of 32 rows). S and O^T are
//    double-buffered in tensor memory. A row of kv head a meets the columns of
//    kv head b too; those products are not used, and P is zero there;
//  - warps 4p..4p+3, softmax (warp w owns tensor-memory lanes 32 (w % 4)..):
//    thread t reads row t of S (page t / 32, kv head (t / 16) % 2, token
//    t % 16) and forms its 4 heads' scores, the exact running max per head
//    (over 16 lanes, then over the 4 warps), the weights and their E4M3 parts;
//    two tiles later it reads row t of O^T (dim t) into its running output of
//    all 8 heads.
//
// Numerics. An E4M3 value has 4 significant bits, bf16 8. q row h is scaled
// by a power of two 2^-e (its largest |q| into [128, 256)) and split as
// q 2^-e = p1 + p2 / 16: p1 is q 2^-e rounded to E4M3 and p2 16 times what is
// left, rounded again, which holds a bf16 q exactly (elements more than 2^14
// below the row's largest keep an error under 2^-21 of it). Column 2h + k of
// the B operand holds part k of q head h of the tile. The weights are
// P = 2^(x - m + 8) <= 256, m the running max (exact per tile: the output
// accumulates in registers, so a rescale costs a multiply), split the same way
// (columns 2h + k): each weight to 2^-9 of itself and 2^-14 absolutely, below
// the rounding of a bf16 output. The tensor cores form the products exactly
// and sum them in f32.
#pragma once

#include <type_traits>

#include "pd_decode_mma.cuh"

namespace pd {

struct CfgTc {
    static constexpr int kD = 128;
    static constexpr int kChunks = 4;                  // pages (16 rows x 2 kv heads) per tile
    static constexpr int kChunkBytes = 2 * kMmaRows * 128;  // one box: 16 rows x 2 kv heads x 128 codes
    static constexpr int kRows = kChunks * 2 * kMmaRows;    // 128 rows per tile: the mma M
    static constexpr int kHeads = 8;                   // q heads per tile (4 per kv head)
    static constexpr int kStages = 3;
    static constexpr int kN = 16;                      // mma N: (head, part) columns of S and of P
    static constexpr int kTileBytes = kRows * 128;     // the E4M3 codes of one K (or V) tile
    static constexpr int kVOff = kTileBytes;
    static constexpr int kQOff = 2 * kTileBytes;       // q parts: kN rows of 128 codes
    static constexpr int kStageBytes = kQOff + kN * 128;
    static constexpr int kPOff = kStages * kStageBytes;  // P parts: two buffers of kN rows of 128 codes
    static constexpr int kMetaOff = kPOff + 2 * kN * 128;
    static constexpr int kMetaInts = 32;               // per stage, see the kMeta* indices
    static constexpr int kRedOff = kMetaOff + kStages * kMetaInts * 4;
    static constexpr int kRedFloats = 2 * 4 * kHeads;  // [tile parity][warp][head]
    static constexpr int kBarOff = kRedOff + 2 * kRedFloats * 4;  // maxima, then sums
    static constexpr int kMiscOff = kBarOff + 24 * 8;  // tensor-memory address, abort flag
    static constexpr int kBytes = kMiscOff + 16;       // one pipeline's shared memory
    static constexpr int kPipeBytes = round_up(kBytes, 1024);
    // Two independent pipelines per block (a kernel that holds tensor memory
    // runs one block per SM), each with its own share, 6 warps and columns.
    static constexpr int kPipes = 2;
    static constexpr int kPipeCols = 4 * kN;           // S[2], O^T[2]
    static constexpr int kTmemCols = kPipes * kPipeCols;
    static constexpr int kThreads = kPipes * 192;
    static_assert(kStageBytes % 1024 == 0 && kPOff % 1024 == 0, "operand tiles stay 1024-byte aligned");
};

// Stage metadata (ints): rows of chunks 0..3, then these.
constexpr int kMetaNck = 8, kMetaFlags = 9, kMetaQrow = 10, kMetaSeg = 11, kMetaKp = 12;
constexpr int kMetaE = 16;  // 8 scale exponents, one per q head of the tile

// Barriers (8 bytes each from CfgTc::kBarOff). kBarRMax (two, by tile parity)
// and kBarRSum: the softmax warps' exchanges of per-warp maxima and sums.
constexpr int kBarFull = 0, kBarEmpty = 3, kBarSFull = 6, kBarSFree = 8, kBarPFull = 10, kBarOFull = 12,
              kBarDone = 14, kBarRMax = 15, kBarRSum = 17;

// Byte offset of code x of row r in a tile of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int r, int x) {
    return uint32_t(r) * 128u + uint32_t(((((x >> 4) ^ r) & 7) << 4) | (x & 15));
}

// The two E4M3 parts of each of two values: codes[k] holds part k of v.x
// (low byte) and of v.y (next byte); part 1 is 16 times what part 0 leaves.
__device__ __forceinline__ void e4m3_split2(float2 v, uint32_t (&codes)[2]) {
    codes[0] = uint32_t(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes[0]), __NV_E4M3);
    __half2 h;
    memcpy(&h, &hr, 4);
    const float2 r = __half22float2(h);
    codes[1] = uint32_t(
        __nv_cvt_float2_to_fp8x2(make_float2((v.x - r.x) * 16.f, (v.y - r.y) * 16.f), __NV_SATFINITE, __NV_E4M3));
}

// Elementwise max of |w| (a pair of bf16) and m (a pair of non-negative bf16).
__device__ __forceinline__ uint32_t abs_max2_bf16(uint32_t m, uint32_t w) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w & 0x7fff7fffu));
    return r;
}

// Wait for phase `parity` of `bar`; false when the CTA is aborting or the
// wait runs out (which sets the abort flag and the status bit). One thread.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* flags) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(flags, kFlagTimeout);
            return false;
        }
    }
}

// The same for a whole warp: true only if every lane's wait succeeded, so
// that the lanes of a warp never part ways on a wait that runs out.
__device__ __forceinline__ bool tc_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* flags) {
    return __all_sync(kFull, tc_wait(bar, parity, abort_flag, flags));
}

// ---- the kernel (set-up and producer below, then mma, softmax and teardown)

template <typename T>
__global__ void __launch_bounds__(CfgTc::kThreads, 1)
    decode_tc_fp8_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    static_assert(std::is_same<T, __nv_bfloat16>::value, "two E4M3 parts hold a bf16 q, not an f16 one");
    using C = CfgTc;
    constexpr float kShift = 8.f;  // P = 2^(x - m + 8) <= 256
    const float kNegInf = -__int_as_float(0x7f800000);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // the staged indptr / last_page_len (a.table_bytes, a multiple of 1024), then the pipelines
    int* s_indptr = reinterpret_cast<int*>(base);
    int* s_lpl = s_indptr + kTableMax + 1;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // warps 0-7: softmax of pipeline wid / 4; 8, 9: producers; 10, 11: mma
    const int pipe = wid < 8 ? wid >> 2 : (wid - 8) & 1;
    uint8_t* smem = base + a.table_bytes + pipe * C::kPipeBytes;
    const uint32_t sbase = smem_u32(smem);
    int* meta = reinterpret_cast<int*>(smem + C::kMetaOff);
    float* red_max = reinterpret_cast<float*>(smem + C::kRedOff);
    float* red_sum = red_max + C::kRedFloats;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(base + a.table_bytes + C::kMiscOff);  // pipeline 0's
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    auto bar = [&](int i) { return sbase + C::kBarOff + 8u * uint32_t(i); };
    const long long unit = (long long)blockIdx.x * C::kPipes + pipe;
    const long long p0 = unit * a.pos_per_warp;
    const long long pend = min(p0 + a.pos_per_warp, a.total_pos);

    // ---- set-up: the table, barriers, zero P buffers (P is zero where no row writes it), tensor memory
    Walk<false> walk(a, s_indptr, s_lpl, p0, pend, lane);
    const int first_page = (wid == 8 || wid == 9) ? walk.prefetch_first() : -1;
    walk.stage_table(s_indptr, s_lpl, [&] {
        if (wid < 8 && (tid & 127) == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(bar(kBarFull + s), 1);
                mbar_init(bar(kBarEmpty + s), 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(kBarSFull + b), 1);
                mbar_init(bar(kBarSFree + b), 4);
                mbar_init(bar(kBarPFull + b), 4);
                mbar_init(bar(kBarOFull + b), 1);
            }
            mbar_init(bar(kBarDone), 1);
            mbar_init(bar(kBarRMax), 4);
            mbar_init(bar(kBarRMax + 1), 4);
            mbar_init(bar(kBarRSum), 4);
            fence_mbar_init();
            *abort_flag = 0;
        }
        if (wid < 8)
            for (int i = tid & 127; i < 2 * C::kN * 128 / 16; i += 128)
                *reinterpret_cast<uint4*>(smem + C::kPOff + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        if (wid == 0) tmem_alloc(smem_u32(tslot), C::kTmemCols);
        if (wid == 8 && lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
    });
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    launch_dependents();
    const uint32_t tmem = *tslot + uint32_t(pipe * C::kPipeCols);

    if (p0 < pend && (wid == 8 || wid == 9)) {
        // ================================================================ producer
        walk.build(p0, first_page);
        const uint64_t policy = l2_evict_first_policy();
        // q parts of the current segment: this lane's 64 codes of row n = lane / 2
        // (q head n / 2 of the tile, part n % 2), dims 64 (lane & 1) ..
        uint4 qp[4] = {};
        int qe = 0;
        int j = 0;
        for (;; ++j) {
            const int s = j % C::kStages;
            // ---- walk the tile before its stage is free: lane c < nck holds chunk c
            int nck = 0, flags = 0, qrow = 0, seg = 0, kp = 0;
            int c_slab = 0, c_row = 0, c_kh2 = 0, c_rows = 0;
            if (a.page_size <= kMmaRows) {
                // One chunk per position: the next listed positions, up to the
                // first segment end, at most kChunks in all.
                while (nck < C::kChunks && walk.seek()) {
                    const unsigned avail = walk.mask & (~0u << walk.cur);
                    const unsigned ends = __ballot_sync(kFull, (walk.e_khf & kSegEnd) != 0) & avail;
                    unsigned take = ends != 0u ? avail & (ends ^ (ends - 1u)) : avail;
                    unsigned over = take;  // the set bits past the first kChunks - nck
                    for (int k = nck; k < C::kChunks && over != 0u; ++k) over &= over - 1u;
                    take &= ~over;
                    const int last = 31 - __clz(take);
                    if (nck == 0) {
                        const int first = __ffs(take) - 1;
                        const int khf = __shfl_sync(kFull, walk.e_khf, first);
                        flags = khf & (kSegStart | kSegComplete);
                        qrow = __shfl_sync(kFull, walk.e_qrow, first);
                        seg = __shfl_sync(kFull, walk.e_seg, first);
                        kp = khf >> kKhShift;
                    }
                    for (unsigned rest = take; rest != 0u; rest &= rest - 1u, ++nck) {
                        const int src = __ffs(rest) - 1;
                        const int sl = __shfl_sync(kFull, walk.e_slab, src);
                        const int rw = __shfl_sync(kFull, walk.e_row, src);
                        const int kf = __shfl_sync(kFull, walk.e_khf, src);
                        const int rr = __shfl_sync(kFull, walk.e_valid, src);
                        if (lane == nck) c_slab = sl, c_row = rw, c_kh2 = 2 * (kf >> kKhShift), c_rows = rr;
                    }
                    walk.cur = last + 1;
                    if ((ends >> last) & 1u) {
                        flags |= kSegEnd;
                        break;
                    }
                }
            } else {
                // Pages of more than 16 rows: chunk by chunk.
                Chunk ck;
                while (nck < C::kChunks && walk.template next<kMmaRows>(&ck)) {
                    if (nck == 0) {
                        flags = ck.flags & (kSegStart | kSegComplete);
                        qrow = ck.qrow;
                        seg = ck.seg;
                        kp = ck.kh;
                    }
                    if (lane == nck) c_slab = ck.slab, c_row = ck.row0, c_kh2 = 2 * ck.kh, c_rows = ck.rows;
                    ++nck;
                    if (ck.flags & kSegEnd) {
                        flags |= kSegEnd;
                        break;
                    }
                }
            }
            const int n = lane >> 1, half = lane & 1;
            if (nck > 0 && (flags & kSegStart)) {
                // E4M3 parts of the segment's 8 q rows, scaled per head by 2^-e
                const int h8 = n >> 1, part = n & 1;
                const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) +
                                                                 (size_t(qrow) + h8) * (C::kD * sizeof(T))) + half * 8;
                uint4 w[8];
                uint32_t mx2 = 0u;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    w[x] = __ldg(qr + x);
                    mx2 = abs_max2_bf16(abs_max2_bf16(mx2, w[x].x), w[x].y);
                    mx2 = abs_max2_bf16(abs_max2_bf16(mx2, w[x].z), w[x].w);
                }
                const float2 m2 = unpack_pair<T>(mx2);
                float mx = fmaxf(m2.x, m2.y);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                qe = mx > 0.f ? max(-100, min(100, ((__float_as_int(mx) >> 23) & 0xff) - 134)) : 0;
                const float inv = __int_as_float((127 - qe) << 23);
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    // codes of dims 64 half + 16 x .. + 15, 4 per word
                    uint32_t cw[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint4& src = w[2 * x + (q4 >> 1)];
                        const uint32_t lo = (q4 & 1) ? src.z : src.x, hi = (q4 & 1) ? src.w : src.y;
                        const float2 a01 = unpack_pair<T>(lo), a23 = unpack_pair<T>(hi);
                        uint32_t c01[2], c23[2];
                        e4m3_split2(make_float2(a01.x * inv, a01.y * inv), c01);
                        e4m3_split2(make_float2(a23.x * inv, a23.y * inv), c23);
                        cw[q4] = ((part ? c01[1] : c01[0]) & 0xffffu) | ((part ? c23[1] : c23[0]) << 16);
                    }
                    qp[x] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                }
            }
            // ---- the stage is free once the P.V of the tile before it has completed
            if (j >= C::kStages &&
                !tc_wait_warp(bar(kBarEmpty + s), uint32_t(j / C::kStages - 1) & 1u, abort_flag, a.flags))
                break;
            const uint32_t st = sbase + uint32_t(s) * C::kStageBytes;
            const uint32_t full = bar(kBarFull + s);
            int* mt = meta + s * C::kMetaInts;
            if (nck == 0) {
                if (lane == 0) {
                    mt[kMetaFlags] = kEndOfWork;
                    mbar_arrive(full);
                }
                ++j;
                break;
            }
            const unsigned copies = __ballot_sync(kFull, lane < nck && c_rows > 0);
            if (lane == 0 && copies != 0u) mbar_expect_tx(full, __popc(copies) * 2u * C::kChunkBytes);
            __syncwarp();
            if (lane < nck) {
                mt[lane] = c_rows;
                if (c_rows > 0) {
                    tma_load_4d(st + lane * C::kChunkBytes, &tmk, 0, c_row, c_kh2, c_slab, full, policy);
                    tma_load_4d(st + C::kVOff + lane * C::kChunkBytes, &tmv, 0, c_row, c_kh2, c_slab, full, policy);
                }
            }
            uint8_t* qa = smem + s * C::kStageBytes + C::kQOff;
#pragma unroll
            for (int x = 0; x < 4; ++x) *reinterpret_cast<uint4*>(qa + sw128_off(n, 64 * half + 16 * x)) = qp[x];
            if ((lane & 3) == 0) mt[kMetaE + (lane >> 2)] = qe;  // lane 4 h holds row 2 h, part 0, of head h
            if (lane == 0) {
                mt[kMetaNck] = nck;
                mt[kMetaFlags] = flags;
                mt[kMetaQrow] = qrow;
                mt[kMetaSeg] = seg;
                mt[kMetaKp] = kp;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // test-only: unit 0's first stage expects bytes that never arrive
                if (j == 0 && unit == 0 && a.test_extra_tx > 0) mbar_expect_tx(full, uint32_t(a.test_extra_tx));
                mbar_arrive(full);
            }
        }
        // The copies of the stages issued last may still be landing when
        // another role has stopped early (all of them have landed otherwise).
        for (int t = max(0, j - C::kStages); t < j; ++t)
            mbar_wait_bounded(bar(kBarFull + t % C::kStages), uint32_t(t / C::kStages) & 1u);
    } else if (p0 < pend && wid >= 10) {
        // ================================================================ mma
        // Issues S of tile jq once its copies have landed and its S buffer is
        // free, and P.V of tile jp once its weights are written, whichever is
        // ready first (a stage is released by its P.V, so P.V does not wait
        // behind the next tile's copies).
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc_idesc_e4m3(C::kRows, C::kN, false);
            constexpr uint32_t idesc_o = tc_idesc_e4m3(C::kRows, C::kN, true);
            int jq = 0, jp = 0, j_end = -1;  // j_end: the end-of-work tile, once seen
            unsigned long long t_idle = global_ns();
            while (j_end < 0 || jp < j_end) {
                bool progress = false;
                if (jp < jq && mbar_test_wait(bar(kBarPFull + (jp & 1)), uint32_t(jp >> 1) & 1u)) {
                    tc_fence_after();
                    const int sp = jp % C::kStages;
                    const uint32_t vt = sbase + uint32_t(sp) * C::kStageBytes + C::kVOff;
                    const uint32_t pb = sbase + C::kPOff + uint32_t(jp & 1) * C::kN * 128;
                    const uint32_t d = tmem + 2 * C::kN + uint32_t(jp & 1) * C::kN;
#pragma unroll
                    for (int k = 0; k < C::kRows / 32; ++k)
                        tc_mma_e4m3(d, smem_desc_sw128(vt + 32 * 128 * k, C::kTileBytes, 1024),
                                    smem_desc_sw128(pb + 32 * k, 16, 1024), idesc_o, k > 0);
                    tc_commit(bar(kBarOFull + (jp & 1)));
                    tc_commit(bar(kBarEmpty + sp));
                    ++jp;
                    progress = true;
                }
                if (j_end < 0 && (jq < 2 || mbar_test_wait(bar(kBarSFree + (jq & 1)), uint32_t((jq - 2) >> 1) & 1u)) &&
                    mbar_test_wait(bar(kBarFull + jq % C::kStages), uint32_t(jq / C::kStages) & 1u)) {
                    const int s = jq % C::kStages;
                    if (meta[s * C::kMetaInts + kMetaFlags] & kEndOfWork) {
                        mbar_arrive(bar(kBarSFull + (jq & 1)));  // the softmax warps see the end too
                        j_end = jq;
                    } else {
                        tc_fence_after();
                        const uint32_t st = sbase + uint32_t(s) * C::kStageBytes;
                        const uint32_t d = tmem + uint32_t(jq & 1) * C::kN;
#pragma unroll
                        for (int k = 0; k < C::kD / 32; ++k)
                            tc_mma_e4m3(d, smem_desc_sw128(st + 32 * k, 16, 1024),
                                        smem_desc_sw128(st + C::kQOff + 32 * k, 16, 1024), idesc_s, k > 0);
                        tc_commit(bar(kBarSFull + (jq & 1)));
                        ++jq;
                    }
                    progress = true;
                }
                if (progress) {
                    t_idle = global_ns();
                } else {
                    __nanosleep(32);  // leave the issue slots to the warps that share the SM
                    if (*abort_flag) break;
                    if (global_ns() - t_idle > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(a.flags, kFlagTimeout);
                        break;
                    }
                }
            }
            // every mma has completed before the tensor memory is released
            tc_commit(bar(kBarDone));
            mbar_wait_bounded(bar(kBarDone), 0u);
        }
    } else if (p0 < pend) {
        // ================================================================ softmax (warps 4p..4p+3)
        const int t = tid & 127;        // row of S (page t / 32, kv head sel, token t % 16); dim row of O^T
        const int sel = (t >> 4) & 1;   // which kv head of the pair row t belongs to
        const uint32_t tl = tmem + (uint32_t(32 * (wid & 3)) << 16);
        float m[8];                     // running max of each q head of the tile (the same in every thread)
        float l[4];                     // this thread's part of the sums of its kv head's 4 q heads
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // running output, dim t, 8 heads
        // The two tiles whose O^T is pending: flags, q row, segment, pair,
        // rescale of the output before the tile is added, and (at a segment
        // end) the maxima and this thread's part of the sums.
        struct Pending {
            int flags, qrow, seg, kp;
            float al[8], m[8], l[4];
        };
        Pending q1{}, q2{};  // tiles j - 1 and j - 2
#pragma unroll
        for (int h = 0; h < 8; ++h) m[h] = kNegInf;
#pragma unroll
        for (int h = 0; h < 4; ++h) l[h] = 0.f;
        int n_sums = 0;  // sum exchanges so far (the phase of kBarRSum)
        // Lanes 0 and 16 of each warp have written their values: arrive, and
        // wait for the other three warps (bounded, unlike a named barrier, so
        // that a warp that stops on an abort cannot leave the others waiting).
        auto exchange = [&](uint32_t b, uint32_t parity) -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(b);
            return tc_wait_warp(b, parity, abort_flag, a.flags);
        };
        // Max (or sum) of v over the 16 lanes of this thread's kv head.
        auto half_max = [&](float v) {
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
            return v;
        };
        auto half_sum = [&](float v) {
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) v += __shfl_xor_sync(kFull, v, off);
            return v;
        };

        // Add O^T of tile jj (state ps) into o; at its segment's end, write the results.
        auto add_o = [&](int jj, const Pending& ps) -> bool {
            if (!tc_wait_warp(bar(kBarOFull + (jj & 1)), uint32_t(jj >> 1) & 1u, abort_flag, a.flags)) return false;
            tc_fence_after();
            uint32_t r[16];
            tmem_ld16(tl + 2 * C::kN + uint32_t(jj & 1) * C::kN, r);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 8; ++h)
                o[h] = fmaf(o[h], ps.al[h], fmaf(__uint_as_float(r[2 * h + 1]), 0.0625f, __uint_as_float(r[2 * h])));
            if (ps.flags & kSegEnd) {
                // the segment's sums: over the 16 lanes of a kv head, then over the warps
                float* rs = red_sum + (jj & 1) * 32;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float v = half_sum(ps.l[h]);
                    if ((lane & 15) == 0) rs[(wid & 3) * 8 + 4 * sel + h] = v;
                }
                if (!exchange(bar(kBarRSum), uint32_t(n_sums++) & 1u)) return false;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float L = (rs[h] + rs[8 + h]) + (rs[16 + h] + rs[24 + h]);
                    const float vsc = __ldg(a.v_scale + 2 * ps.kp + (h >> 2));
                    const float inv = L > 0.f ? vsc / L : 0.f;
                    const float lse = L > 0.f ? ps.m[h] - kShift + log2f(L) : kNegInf;
                    if (ps.flags & kSegComplete) {
                        static_cast<T*>(a.o)[(size_t(ps.qrow) + h) * C::kD + t] = T(o[h] * inv);
                        if (t == 0 && a.lse != nullptr) a.lse[size_t(ps.qrow) + h] = lse == kNegInf ? kNegInf : lse * kLn2;
                    } else {
                        const long long slot = unit + ps.seg;
                        a.part_o[(size_t(slot) * 8 + h) * C::kD + t] = o[h] * inv;
                        if (t == 0) a.part_lse[size_t(slot) * 8 + h] = lse;
                    }
                    o[h] = 0.f;
                }
            }
            return true;
        };

        for (int j = 0;; ++j) {
            const int s = j % C::kStages;
            if (!tc_wait_warp(bar(kBarSFull + (j & 1)), uint32_t(j >> 1) & 1u, abort_flag, a.flags)) break;
            if (!tc_wait_warp(bar(kBarFull + s), uint32_t(j / C::kStages) & 1u, abort_flag, a.flags)) break;
            const int* mt = meta + s * C::kMetaInts;
            const int flags = mt[kMetaFlags];
            if (flags & kEndOfWork) {
                if (j >= 2 && !add_o(j - 2, q2)) break;
                if (j >= 1) add_o(j - 1, q1);
                break;
            }
            // ---- scores of row t: its kv head's 4 q heads (columns 8 sel + 2h + part)
            tc_fence_after();
            uint32_t r[16];
            tmem_ld16(tl + uint32_t(j & 1) * C::kN, r);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + (j & 1)));
            const int c = t >> 5;
            const bool valid = c < mt[kMetaNck] && (t & 15) < mt[c];
            const int kp = mt[kMetaKp];
            const float qs = a.q_scale * __ldg(a.k_scale + 2 * kp + sel);
            float x[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float s0 = __uint_as_float(sel ? r[8 + 2 * h] : r[2 * h]);
                const float s1 = __uint_as_float(sel ? r[9 + 2 * h] : r[2 * h + 1]);
                const float sc = qs * __int_as_float((127 + mt[kMetaE + 4 * sel + h]) << 23);
                x[h] = valid ? fmaf(s1, 0.0625f, s0) * sc : kNegInf;
            }
            // ---- the tile's max per q head: 16 lanes, then the 4 warps
            float* rm = red_max + (j & 1) * 32;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float v = half_max(x[h]);
                if ((lane & 15) == 0) rm[(wid & 3) * 8 + 4 * sel + h] = v;
            }
            if (!exchange(bar(kBarRMax + (j & 1)), uint32_t(j >> 1) & 1u)) break;
            if (flags & kSegStart) {
#pragma unroll
                for (int h = 0; h < 8; ++h) m[h] = kNegInf;
#pragma unroll
                for (int h = 0; h < 4; ++h) l[h] = 0.f;
            }
            Pending cur;
            cur.flags = flags;
            cur.qrow = mt[kMetaQrow];
            cur.seg = mt[kMetaSeg];
            cur.kp = kp;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float tm = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
                const float mn = fmaxf(m[h], tm);
                cur.al[h] = m[h] == kNegInf ? 0.f : ex2(m[h] - mn);
                m[h] = mn;
                cur.m[h] = mn;
            }
            float p[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float ms = sel ? m[4 + h] : m[h];
                const float as = sel ? cur.al[4 + h] : cur.al[h];
                p[h] = x[h] == kNegInf ? 0.f : ex2(x[h] - ms + kShift);
                l[h] = fmaf(l[h], as, p[h]);
                cur.l[h] = l[h];
            }
            // ---- a row past the valid rows must not hold a NaN code under a zero weight
            if (!valid) {
                uint4* vr = reinterpret_cast<uint4*>(smem + s * C::kStageBytes + C::kVOff + t * 128);
#pragma unroll
                for (int x8 = 0; x8 < 8; ++x8) vr[x8] = make_uint4(0u, 0u, 0u, 0u);
            }
            // ---- O^T of tile j - 2 (it read the P buffer this tile writes)
            if (j >= 2 && !add_o(j - 2, q2)) break;
            // ---- the E4M3 parts of P: row 2 (4 sel + h) + part of the B operand, code t
            uint8_t* pb = smem + C::kPOff + (j & 1) * C::kN * 128;
#pragma unroll
            for (int h = 0; h < 4; h += 2) {
                uint32_t cd[2];
                e4m3_split2(make_float2(p[h], p[h + 1]), cd);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    pb[sw128_off(8 * sel + 2 * h + k, t)] = uint8_t(cd[k] & 0xffu);
                    pb[sw128_off(8 * sel + 2 * (h + 1) + k, t)] = uint8_t((cd[k] >> 8) & 0xffu);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPFull + (j & 1)));
            q2 = q1;
            q1 = cur;
        }
    }

    // ---- teardown: every role is done with the tensor memory
    tc_fence_before();
    __syncthreads();
    if (wid == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(*tslot, C::kTmemCols);
    }
}

}  // namespace pd
