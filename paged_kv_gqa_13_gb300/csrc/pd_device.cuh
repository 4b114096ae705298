// Device-side building blocks shared by the pagedecode kernels: PTX wrappers
// for mbarriers, bulk async copies and programmatic dependent launch, element
// conversions, warp reductions and the kernel argument blocks.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pd {

// Status word bits (the same values as PD_FLAG_* in pagedecode.h).
constexpr int kFlagBadPage = 0x1;
constexpr int kFlagBadLastPageLen = 0x2;
constexpr int kFlagBadIndptr = 0x4;
constexpr int kFlagTimeout = 0x8;

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// Upper bound on one pipeline wait. Copies of a few KB finish in
// microseconds; this only ends a wait that can never finish.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy global stores before async-proxy
// (bulk copy / TMA) reads issued after it (and after a warp barrier, by
// another lane of the warp).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test for the completion of phase `parity` of a barrier.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of a barrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk async copy global -> shared, completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (no shared memory, no
// completion). src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 4-D tiled tensor copy global -> shared through a tensor map (TMA), with
// completion counted in bytes on `bar`. The innermost coordinate c0 is in
// elements; c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int c0, int c1, int c2, int c3,
                                           uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Four 8x8 b16 matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8. Lane l receives row l / 4, elements 2(l % 4) and
// 2(l % 4) + 1 of each matrix (the mma fragment layout).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// The same, each matrix delivered transposed.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held in the mma fragment layout.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D += A * B for one m16n8k16 tile, 16-bit inputs of type T, f32 accumulate.
template <typename T>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma_16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma_16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9},"
        " {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- tcgen05 (5th-generation tensor cores)

// Allocate `ncols` columns (a power of two, 32..512) of tensor memory for this
// CTA, all 128 lanes; the whole warp calls it and the address (lane 0, first
// column) lands at dst (shared memory). Freed by tmem_dealloc, by one warp,
// before the CTA exits.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations before / after a thread synchronisation (a
// barrier or an mbarrier wait) that hands tensor memory from thread to thread.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on the mbarrier at `bar` when every tcgen05.mma this thread has
// issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor of an operand tile in the 128-byte swizzle
// layout: rows of 128 bytes, 16-byte piece x of row r at piece x ^ (r & 7),
// 8-row groups of 1024 bytes. For a K-major operand the rows are the M (or N)
// index, `sbo` the step between 8-row groups and `lbo` unused; for an
// MN-major one the rows are the K index, `sbo` the step between groups of 8
// K rows and `lbo` the step between 128-byte blocks along M (N). addr must be
// 1024-byte aligned, or advanced from such an address by less than 128 bytes
// along a K-major row (one k step).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr >> 4) & 0x3fffu) | (uint64_t((lbo >> 4) & 0x3fffu) << 16) |
           (uint64_t((sbo >> 4) & 0x3fffu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B and
// an f32 accumulator, for an M x N tile; a_mn: A is MN-major.
__host__ __device__ constexpr uint32_t tc_idesc_e4m3(int M, int N, bool a_mn) {
    return (1u << 4) | (a_mn ? 1u << 15 : 0u) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D (tensor memory) = A * B (+ D when acc), A and B E4M3 from shared memory.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(uint32_t(acc))
        : "memory");
}

// 16 consecutive f32 columns of one tensor-memory lane per thread: thread l
// of the warp reads lane (taddr >> 16) + l. A warp may read only the 32
// lanes 32 (warp % 4) ..; followed by tmem_wait_ld before the values are used.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Raise the transaction count of the current phase of `bar` by `bytes`
// (without arriving).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// 2^x on the special-function unit; inputs far below 0 give +0, -inf gives +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- elements

// Eight E4M3 codes (little-endian bytes of w) to f32. Every E4M3 value is an
// f16 value, so the two steps through f16 are exact.
__device__ __forceinline__ void e4m3x8_to_f32(uint2 w, float* f) {
    const uint32_t h[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __half2_raw r =
                __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(h[i] >> (16 * j)), __NV_E4M3);
            __half2 v;
            memcpy(&v, &r, 4);
            const float2 x = __half22float2(v);
            f[4 * i + 2 * j] = x.x;
            f[4 * i + 2 * j + 1] = x.y;
        }
    }
}

// Two E4M3 codes (the low 16 bits of w, first code in the low byte) to an
// f16x2 word, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
    uint32_t out;
    memcpy(&out, &r, 4);
    return out;
}

template <typename T>
struct Elt;

template <>
struct Elt<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ void to_f32(const uint4& r, float* f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
    __device__ static __forceinline__ uint4 from_f32(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

template <>
struct Elt<__half> {
    static constexpr int kVec = 8;
    __device__ static __forceinline__ float2 pair(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    __device__ static __forceinline__ void to_f32(const uint4& r, float* f) {
        float2 a = pair(r.x), b = pair(r.y), c = pair(r.z), d = pair(r.w);
        f[0] = a.x, f[1] = a.y, f[2] = b.x, f[3] = b.y, f[4] = c.x, f[5] = c.y, f[6] = d.x, f[7] = d.y;
    }
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ static __forceinline__ uint4 from_f32(const float* f) {
        return make_uint4(pack(f[0], f[1]), pack(f[2], f[3]), pack(f[4], f[5]), pack(f[6], f[7]));
    }
};

template <>
struct Elt<__nv_bfloat16> {
    static constexpr int kVec = 8;
    // A bfloat16 is the upper half of a float: widening is a shift or a mask.
    __device__ static __forceinline__ void to_f32(const uint4& r, float* f) {
        f[0] = __uint_as_float(r.x << 16), f[1] = __uint_as_float(r.x & 0xffff0000u);
        f[2] = __uint_as_float(r.y << 16), f[3] = __uint_as_float(r.y & 0xffff0000u);
        f[4] = __uint_as_float(r.z << 16), f[5] = __uint_as_float(r.z & 0xffff0000u);
        f[6] = __uint_as_float(r.w << 16), f[7] = __uint_as_float(r.w & 0xffff0000u);
    }
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ static __forceinline__ uint4 from_f32(const float* f) {
        return make_uint4(pack(f[0], f[1]), pack(f[2], f[3]), pack(f[4], f[5]), pack(f[6], f[7]));
    }
};

// ---------------------------------------------------------------- warp reductions

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

// Reduce-scatter of N partial sums across the lanes that differ in the bits
// below 2*OFF (a "row group"). At each level the lane keeps half of its
// values and adds the partner's copy of that half; once one value is left the
// remaining levels are plain butterflies. Total shuffles: N/2 + N/4 + ... per
// lane instead of N * log2(lanes) for N separate all-reduces.
template <int N, int OFF>
struct ReduceScatter {
    __device__ static __forceinline__ void run(float* v, int lane) {
        if constexpr (OFF == 0) {
            return;
        } else if constexpr (N >= 2) {
            constexpr int H = N / 2;
            const bool up = (lane & OFF) != 0;
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float send = up ? v[j] : v[j + H];
                const float keep = up ? v[j + H] : v[j];
                v[j] = keep + __shfl_xor_sync(kFull, send, OFF);
            }
            ReduceScatter<H, OFF / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], OFF);
            ReduceScatter<1, OFF / 2>::run(v, lane);
        }
    }
    // Which of the original N values v[j] holds after run().
    __device__ static __forceinline__ int index(int j, int lane) {
        if constexpr (OFF == 0 || N < 2) {
            return j;
        } else {
            return ReduceScatter<N / 2, OFF / 2>::index(j, lane) + (((lane & OFF) != 0) ? N / 2 : 0);
        }
    }
};

// Reduce-scatter of N float2 values across the lanes that differ in the bits
// OFF, OFF/2, ..., STOP (lane bits of the row groups): after it a lane holds
// N / (OFF*2/STOP) complete sums, those of the indices given by index().
template <int N, int OFF, int STOP>
struct ReduceScatter2 {
    __device__ static __forceinline__ void run(float2* v, int lane) {
        if constexpr (OFF < STOP || OFF == 0) {
            return;
        } else {
            static_assert(N >= 2, "one value per lane is the finest split");
            constexpr int H = N / 2;
            const bool up = (lane & OFF) != 0;
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float2 send = up ? v[j] : v[j + H];
                const float2 keep = up ? v[j + H] : v[j];
                const float2 got = make_float2(__shfl_xor_sync(kFull, send.x, OFF), __shfl_xor_sync(kFull, send.y, OFF));
                v[j] = __fadd2_rn(keep, got);
            }
            ReduceScatter2<H, OFF / 2, STOP>::run(v, lane);
        }
    }
    __device__ static __forceinline__ int index(int j, int lane) {
        if constexpr (OFF < STOP || OFF == 0) {
            return j;
        } else {
            return ReduceScatter2<N / 2, OFF / 2, STOP>::index(j, lane) + (((lane & OFF) != 0) ? N / 2 : 0);
        }
    }
};

// ---------------------------------------------------------------- arguments

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* indices;
    const int32_t* indptr;
    const int32_t* last_page_len;
    void* o;
    float* lse;       // may be null (contiguous entry)
    float* part_o;    // [slots][G][D] f32, normalised partial outputs
    float* part_lse;  // [slots][G] f32, partial lse in log2 units
    int* flags;       // sticky status word
    int batch, num_qo_heads, num_kv_heads, page_size, num_total_pages;
    int group, head_tiles, heads_per_tile;
    int n_pos;                 // positions per (kv head, head tile) pass
    int table_bytes;           // dynamic smem bytes holding the staged indptr/last_page_len
    long long total_pos;       // head_tiles * num_kv_heads * n_pos
    long long pos_per_warp;
    float q_scale;             // sm_scale * log2(e)
    int contiguous;            // 0: paged store, 1: contiguous cache
    long long slab_rows;       // rows from one (page | request, kv head) slab to the next:
                               // page_size (paged) or max_kv_len (contiguous)
    int valid_kv_len, vpage, npv;  // contiguous: valid rows, rows per virtual page, pages per request
    // Fused append (null otherwise): [batch, num_kv_heads, D] rows that become
    // the last valid row of every (request, kv head) before it is read. The
    // kernel then writes into k and v.
    const void* k_new;
    const void* v_new;
    // FP8 pools (null otherwise): element value = E4M3 code value * scale[kv head].
    const float* k_scale;
    const float* v_scale;
    int test_extra_tx;  // test-only wait-timeout injection (pd_test_inject_wait_timeout); normally 0
    // 0: warp w of block c holds unit c * warps_per_block + w. 1: unit
    // w * blocks + c, with one pass per warp of a block and passes padded to a
    // whole number of units, so that a block's warps hold the same token range
    // of every pass (token-major contiguous cache).
    int unit_transpose;
    // Positions at the end of each warp's share (pos_per_warp) that its warp
    // does not run (0: none): they are cut into tail_pieces units (the last
    // takes the remainder), handed out in share order to warps that have
    // finished their own range. Share s is units (1 + k) s (head, its warp)
    // and (1 + k) s + 1 .. (1 + k) s + k (tail pieces, any warp), k =
    // tail_pieces. The unit boundaries are fixed, so the results do not
    // depend on which warp runs a piece. tail_ctl (workspace header): [0]
    // next piece, [1] warps finished; the last warp of the grid to finish
    // sets both back to zero.
    int tail;
    int tail_pieces;
    unsigned* tail_ctl;
};

struct MergeArgs {
    const float* part_o;
    const float* part_lse;
    const int32_t* indptr;
    void* o;
    float* lse;
    int* flags;
    int batch, num_qo_heads, num_kv_heads, group, head_tiles, heads_per_tile, G;
    int n_pos;
    long long pos_per_warp;
    int contiguous, npv;
    int append;  // fused append: a request with no page is an error (flagged)
    int tail, tail_pieces;  // DecodeArgs::tail, tail_pieces of the decode that wrote the partials
};

// Position range [lo, hi) of request b within one pass over the positions.
// Shared by the decode walk and the merge so that both cut identically.
__device__ __forceinline__ void request_range(int b, int n_pos, bool contiguous, int npv, int raw_lo,
                                              int raw_hi, int* lo, int* hi) {
    if (contiguous) {
        *lo = b * npv;
        *hi = (b + 1) * npv;
        return;
    }
    int l = raw_lo < 0 ? 0 : (raw_lo > n_pos ? n_pos : raw_lo);
    int h = raw_hi > n_pos ? n_pos : raw_hi;
    *lo = l;
    *hi = h < l ? l : h;
}

}  // namespace pd
