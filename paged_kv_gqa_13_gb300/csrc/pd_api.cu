// The C ABI of pagedecode: argument checks, planning of the work partition,
// kernel launches, the paged append and copy kernels, profiling hooks.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pagedecode.h"
#include "pd_kernels.cuh"

namespace pd {
bool lookup_kernels_f32(int head_dim, int heads, KernelSet* ks);
bool lookup_kernels_f16(int head_dim, int heads, KernelSet* ks);
bool lookup_kernels_bf16(int head_dim, int heads, KernelSet* ks);
#define PD_VARIANTS(dt)                                                    \
    bool lookup_fused_##dt(int head_dim, int heads, const void** fn);      \
    bool lookup_nhd_##dt(int head_dim, int heads, const void** fn);        \
    bool lookup_nhd_fused_##dt(int head_dim, int heads, const void** fn);
PD_VARIANTS(f32)
PD_VARIANTS(f16)
PD_VARIANTS(bf16)
#undef PD_VARIANTS
bool lookup_fp8_f16(int head_dim, int heads, bool kv_pairs, KernelSet* ks);
bool lookup_fp8_bf16(int head_dim, int heads, bool kv_pairs, KernelSet* ks);
}  // namespace pd

namespace {

thread_local char g_err[512] = "";

pd_status fail(pd_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pd_status fail(pd_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

pd_status ok() {
    g_err[0] = '\0';
    return PD_OK;
}

pd_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(pd_dtype dt) { return dt == PD_F32 ? 4 : 2; }

bool lookup(pd_dtype dt, int D, int G, pd::KernelSet* ks) {
    switch (dt) {
#define PD_LOOKUP(dt)                                                                                  \
    if (!pd::lookup_kernels_##dt(D, G, ks)) return false;                                               \
    ks->variant[0] = ks->decode;                                                                        \
    return pd::lookup_fused_##dt(D, G, &ks->variant[1]) && pd::lookup_nhd_##dt(D, G, &ks->variant[2]) && \
           pd::lookup_nhd_fused_##dt(D, G, &ks->variant[3]);
        case PD_F32: { PD_LOOKUP(f32) }
        case PD_F16: { PD_LOOKUP(f16) }
        case PD_BF16: { PD_LOOKUP(bf16) }
#undef PD_LOOKUP
    }
    return false;
}

// Kernels for an E4M3 pool with q / o of type dt (f16 or bf16).
// pd_select_fp8_kernel: 1 when the tcgen05 E4M3 kernel is chosen where it applies.
std::atomic<int> g_fp8_tcgen05{0};

bool kv_pairs_ok(pd_dtype dt, int Hq, int Hk) {
    return g_fp8_tcgen05.load(std::memory_order_relaxed) != 0 && dt == PD_BF16 && Hk % 2 == 0 && Hq == 4 * Hk;
}

// kv_pairs: the shape allows the kernel that takes the kv heads in pairs (bf16,
// groups of exactly 4 q heads, an even number of kv heads).
bool lookup_fp8(pd_dtype dt, int D, int G, bool kv_pairs, pd::KernelSet* ks) {
    switch (dt) {
        case PD_F16: return pd::lookup_kernels_f16(D, G, ks) && pd::lookup_fp8_f16(D, G, kv_pairs, ks);
        case PD_BF16: return pd::lookup_kernels_bf16(D, G, ks) && pd::lookup_fp8_bf16(D, G, kv_pairs, ks);
        default: return false;
    }
}

// Per-device facts, read once.
struct DeviceInfo {
    int sms = 0;
    int max_smem = 0;
};

std::mutex g_mu;

pd_status device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static std::vector<DeviceInfo> cache;
    std::lock_guard<std::mutex> lk(g_mu);
    if (int(cache.size()) <= dev) cache.resize(dev + 1);
    if (cache[dev].sms == 0) {
        int sms = 0, smem = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        cache[dev].sms = sms;
        cache[dev].max_smem = smem;
    }
    *out = cache[dev];
    return PD_OK;
}

// Raise a kernel's dynamic shared memory limit once per (device, kernel, size).
pd_status allow_smem(const void* fn, int bytes) {
    int dev = 0;
    cudaGetDevice(&dev);
    struct Entry {
        int dev;
        const void* fn;
        int bytes;
    };
    static std::vector<Entry> done;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (const Entry& x : done)
            if (x.dev == dev && x.fn == fn && x.bytes >= bytes) return PD_OK;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    std::lock_guard<std::mutex> lk(g_mu);
    done.push_back({dev, fn, bytes});
    return PD_OK;
}

// How a decode call is laid out on the device.
// Dynamic tails (DecodeArgs::tail): shares of at least kTailMinPos positions
// give their last 1/kTailDiv (1/kTailDivShort for shares of at most
// kShortShareRows rows), in kTailPieces pieces, to whichever warps finish
// first; a share's length is counted in K/V rows (positions x rows per page or
// virtual page). The counters sit in the workspace header after the status word. A
// plan holds 1 + kTailMaxPieces partial slots per warp.
// Measured on GB300, tails claimed ahead, same box: the 32-request Llama-shaped
// batch (~33 pages of 16 rows per share, 528 rows) takes 64.1 / 62.4 / 62.2 us
// per call with tails of 1/8, 1/3 and 1/4; batches with shares of ~3,000-3,500
// rows (ragged 70B, long context paged and contiguous, MHA) are fastest at 1/8
// and lose 2.5-5 % at 1/5 or 1/4. Earlier, tails of 1/4 .. 1/6 cut in two pieces shortened the long
// batches by ~1 % but cost more than that in the merge of the 32-request batch.
constexpr long long kTailMinPos = 12;
constexpr long long kTailDiv = 8;
constexpr long long kShortShareRows = 1024;
constexpr long long kTailDivShort = 4;
constexpr int kTailPieces = 1;
constexpr int kTailMaxPieces = 1;
constexpr size_t kTailCtlOff = 64;

struct Plan {
    int group = 0, head_tiles = 0, heads_per_tile = 0, G = 0;
    pd::KernelSet ks{};
    int table_bytes = 0, nwarps = 0, ctas = 0, sms = 0;
    long long total_warps = 0, segments = 0, slots = 0;
    int walk_kv = 0;     // kv heads as the walk and the merge see them: Hk, or Hk / 2 pairs (ks.mma 3)
    bool tails = false;  // the decode kernel takes DecodeArgs::tail (slots for two units per warp)
    size_t smem = 0, lse_off = 0, o_off = 0, ws_bytes = 0;
};

// Threads per decode block: one warp per share, or the kernel's own block
// when its shares are groups of warps.
int block_threads(const Plan& p) { return p.ks.threads > 0 ? p.ks.threads : p.nwarps * 32; }

// Smallest number of head tiles that splits the group into tiles of <= 8 heads.
void split_group(int g, int* tiles, int* per) {
    int t = 1;
    while (g / t > 8 || g % t != 0) ++t;
    *tiles = t;
    *per = g / t;
}

pd_status make_plan_uncached(pd_dtype dt, int batch, int Hq, int Hk, int D, bool contiguous, bool fp8, Plan* p);

// Plans depend only on the shape and the device: keep the last few so that a
// decode loop pays the occupancy query and the attribute set-up once.
// fp8: the K/V pool holds E4M3 codes (dt is then the type of q and o).
pd_status make_plan(pd_dtype dt, int batch, int Hq, int Hk, int D, bool contiguous, Plan* p, bool fp8 = false) {
    struct Entry {
        int dev;
        pd_dtype dt;
        int batch, Hq, Hk, D;
        bool contiguous, fp8, tcgen05;
        Plan plan;
    };
    static Entry cache[16];
    static int used = 0, next = 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    const bool tcgen05 = g_fp8_tcgen05.load(std::memory_order_relaxed) != 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < used; ++i) {
            const Entry& e = cache[i];
            if (e.dev == dev && e.dt == dt && e.batch == batch && e.Hq == Hq && e.Hk == Hk && e.D == D &&
                e.contiguous == contiguous && e.fp8 == fp8 && e.tcgen05 == tcgen05) {
                *p = e.plan;
                return PD_OK;
            }
        }
    }
    const pd_status st = make_plan_uncached(dt, batch, Hq, Hk, D, contiguous, fp8, p);
    if (st != PD_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    cache[next] = Entry{dev, dt, batch, Hq, Hk, D, contiguous, fp8, tcgen05, *p};
    next = (next + 1) % 16;
    if (used < 16) ++used;
    return PD_OK;
}

pd_status make_plan_uncached(pd_dtype dt, int batch, int Hq, int Hk, int D, bool contiguous, bool fp8, Plan* p) {
    if (dt != PD_F32 && dt != PD_F16 && dt != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (batch <= 0 || Hq <= 0 || Hk <= 0) return fail(PD_ERR_INVALID, "batch, num_qo_heads and num_kv_heads must be positive");
    if (Hq % Hk != 0) return fail(PD_ERR_INVALID, "num_qo_heads (%d) must be a multiple of num_kv_heads (%d)", Hq, Hk);
    if (D != 64 && D != 128 && D != 256) return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", D);
    p->group = Hq / Hk;
    split_group(p->group, &p->head_tiles, &p->heads_per_tile);
    p->G = 1;
    while (p->G < p->heads_per_tile) p->G *= 2;
    if (fp8 && dt == PD_F32) return fail(PD_ERR_UNSUPPORTED, "E4M3 pools take f16 or bf16 q and o");
    if (!(fp8 ? lookup_fp8(dt, D, p->G, kv_pairs_ok(dt, Hq, Hk), &p->ks) : lookup(dt, D, p->G, &p->ks)))
        return fail(PD_ERR_UNSUPPORTED, "no kernel for head_dim %d, %d heads per tile", D, p->G);
    p->G = p->ks.part_heads;  // the partial-result layout of the chosen kernel
    p->walk_kv = Hk;
    if (p->ks.mma == 3) {
        // kv heads in pairs: a pair and its 8 q heads are one kv head of group 8
        p->walk_kv = Hk / 2;
        p->group *= 2;
        p->heads_per_tile *= 2;
    }
    DeviceInfo di;
    pd_status st = device_info(&di);
    if (st != PD_OK) return st;
    p->table_bytes = pd::table_bytes_for(!contiguous && batch <= pd::kTableMax);
    p->nwarps = (di.max_smem - p->table_bytes - p->ks.smem_slack) / p->ks.warp_bytes;
    if (p->nwarps > p->ks.max_warps) p->nwarps = p->ks.max_warps;
    if (p->nwarps < 1 || (p->ks.threads > 0 && p->nwarps != p->ks.max_warps))
        return fail(PD_ERR_UNSUPPORTED, "shared memory per block too small for this shape");
    p->smem = size_t(p->ks.smem_slack) + size_t(p->table_bytes) + size_t(p->nwarps) * p->ks.warp_bytes;
    // The variants this plan may launch (NHD only on the contiguous cache) all
    // share its layout; size one wave by the lowest of their occupancies.
    int per_sm = 1 << 30;
    for (int v = 0; v < (contiguous ? 4 : 2); ++v) {
        if (p->ks.variant[v] == nullptr) continue;
        if ((st = allow_smem(p->ks.variant[v], int(p->smem))) != PD_OK) return st;
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, p->ks.variant[v], block_threads(*p), p->smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (n < per_sm) per_sm = n;
    }
    if (per_sm < 1) per_sm = 1;
    p->ctas = di.sms * per_sm;
    p->sms = di.sms;
    p->total_warps = (long long)p->ctas * p->nwarps;
    p->segments = (long long)p->head_tiles * p->walk_kv * batch;
    // All but the E4M3 tensor-core kernels: on the Llama-shaped batch the
    // mma.sync one's shares are ~22 positions, so a tail is one two-page
    // stage, and tails made it slower (36 -> 43 us; with the tails claimed
    // ahead, 36.0 -> 46.3 us); the tcgen05 one has one share per block.
    p->tails = p->ks.mma < 2;
    p->slots = (p->tails ? 1 + kTailMaxPieces : 1) * p->total_warps + p->segments;
    p->lse_off = PD_WORKSPACE_HEADER_BYTES;
    p->o_off = p->lse_off + (size_t(p->slots) * p->G * 4 + 255) / 256 * 256;
    p->ws_bytes = p->o_off + size_t(p->slots) * p->G * D * 4;
    return PD_OK;
}

// ---------------------------------------------------------------- tensor maps

// The driver's tensor-map encoder, reached through the runtime so that the
// library needs no link against the driver library.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// K or V as a 4-D tensor {head_dim, rows, kv heads, slabs} (HND) or
// {head_dim, kv heads, rows, slabs} (NHD). `rows` is the extent read (page
// size, or the valid length of a contiguous cache), `slab_rows` the rows
// allocated per (slab, kv head) that set the strides; rows past `rows` read as
// zero. mma 1: boxes of 64 16-bit columns x 16 rows with the 128-byte
// swizzle (the tensor-core kernel); mma 2: the same for E4M3 codes, 128
// one-byte columns (the E4M3 tensor-core kernel). mma 0: unswizzled boxes of
// head_dim columns x `box_rows` rows (the CUDA-core kernel on an NHD cache).
// A box holds rows of one kv head, so it lands as consecutive rows either way.
pd_status make_kv_map(CUtensorMap* map, const void* base, pd_dtype dt, int D, long long rows, long long slab_rows,
                      int Hk, long long slabs, bool nhd, int mma, int box_rows, int box_heads = 1) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return fail(PD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    // mma 2: E4M3 codes, one byte per element, whatever the type of q and o
    const cuuint64_t row = cuuint64_t(D) * (mma == 2 ? 1u : elem_size(dt));
    const cuuint64_t dims_hnd[4] = {cuuint64_t(D), cuuint64_t(rows), cuuint64_t(Hk), cuuint64_t(slabs)};
    const cuuint64_t dims_nhd[4] = {cuuint64_t(D), cuuint64_t(Hk), cuuint64_t(rows), cuuint64_t(slabs)};
    const cuuint64_t str_hnd[3] = {row, cuuint64_t(slab_rows) * row, cuuint64_t(Hk) * slab_rows * row};
    const cuuint64_t str_nhd[3] = {row, cuuint64_t(Hk) * row, cuuint64_t(Hk) * slab_rows * row};
    const cuuint64_t* dims = nhd ? dims_nhd : dims_hnd;
    const cuuint64_t* strides = nhd ? str_nhd : str_hnd;
    // a swizzled box row is 128 bytes: 64 16-bit or 128 E4M3 elements
    const cuuint32_t cols = mma == 2 ? 128u : mma ? 64u : cuuint32_t(D);
    const cuuint32_t brows = mma ? cuuint32_t(pd::kMmaRows) : cuuint32_t(box_rows);
    const cuuint32_t box_hnd[4] = {cols, brows, cuuint32_t(box_heads), 1};
    const cuuint32_t box_nhd[4] = {cols, 1, brows, 1};
    const cuuint32_t* box = nhd ? box_nhd : box_hnd;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType ty = mma == 2        ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dt == PD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dt == PD_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUresult r = enc(map, ty, 4, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return PD_OK;
}

// ---------------------------------------------------------------- profiling

struct Profile {
    bool on = false;
    std::vector<cudaEvent_t> free_events;
    std::vector<cudaEvent_t> decode_marks;  // pairs: start, end
    std::vector<cudaEvent_t> merge_marks;
    std::vector<cudaEvent_t> append_marks;
};
Profile g_prof;
std::mutex g_prof_mu;

cudaEvent_t take_event() {
    if (g_prof.free_events.empty()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        return e;
    }
    cudaEvent_t e = g_prof.free_events.back();
    g_prof.free_events.pop_back();
    return e;
}

void mark(std::vector<cudaEvent_t>* v, cudaStream_t s) {
    cudaEvent_t e = take_event();
    if (e != nullptr) {
        cudaEventRecord(e, s);
        v->push_back(e);
    }
}

// ---------------------------------------------------------------- decode launch

// Test-only: extra bytes warp 0's first pipeline stage waits for (0: off).
std::atomic<int> g_inject_extra_tx{0};

// nhd: the contiguous cache is token-major, [slabs, slab_rows, Hk, D].
pd_status launch_decode(const Plan& pl, pd::DecodeArgs& a, int D, pd_dtype dt, long long slabs, bool nhd,
                        cudaStream_t stream) {
    const int variant = (a.k_new != nullptr ? pd::kVarFused : 0) | (nhd ? pd::kVarNhd : 0);
    a.test_extra_tx = g_inject_extra_tx.load(std::memory_order_relaxed);
    // Every decode kernel takes two tensor maps; they are read by the
    // tensor-core kernel and by the CUDA-core kernel's NHD variants.
    CUtensorMap maps[2];
    std::memset(maps, 0, sizeof(maps));
    if ((pl.ks.mma || nhd) && a.total_pos > 0) {
        const long long rows = a.contiguous ? a.valid_kv_len : a.slab_rows;
        // both E4M3 kernels take 128-code boxes; the tcgen05 one two kv heads per box
        const int mma = pl.ks.mma == 3 ? 2 : pl.ks.mma;
        const int box_heads = pl.ks.mma == 3 ? 2 : 1;
        pd_status st = make_kv_map(&maps[0], a.k, dt, D, rows, a.slab_rows, a.num_kv_heads, slabs, nhd, mma,
                                   pl.ks.rows_per_stage, box_heads);
        if (st == PD_OK)
            st = make_kv_map(&maps[1], a.v, dt, D, rows, a.slab_rows, a.num_kv_heads, slabs, nhd, mma,
                             pl.ks.rows_per_stage, box_heads);
        if (st != PD_OK) return st;
    }
    std::unique_lock<std::mutex> plk(g_prof_mu);
    const bool prof = g_prof.on;
    if (!prof) plk.unlock();
    cudaError_t e;
    if (a.total_pos > 0) {
        const long long passes = a.total_pos / a.n_pos;
        int grid;
        if (nhd && passes == pl.nwarps && (long long)a.n_pos + pl.ctas <= 0x7fffffffLL) {
            // Token-major cache: block c's warp k takes range c of pass k, so
            // that one SM reads all kv heads of a token range at about the same
            // time (each kv head's rows are 256 B pieces of every token block).
            // Passes are padded to whole units; padding positions hold no request.
            const long long w = pl.ctas;
            a.pos_per_warp = (a.n_pos + w - 1) / w;
            a.n_pos = int(w * a.pos_per_warp);
            a.total_pos = passes * a.n_pos;
            a.unit_transpose = 1;
            grid = int(w);
        } else {
            a.pos_per_warp = (a.total_pos + pl.total_warps - 1) / pl.total_warps;
            const long long warps_used = (a.total_pos + a.pos_per_warp - 1) / a.pos_per_warp;
            grid = int((warps_used + pl.nwarps - 1) / pl.nwarps);
        }
        // SMs stream at different rates (by up to ~25% across one GPU), so
        // equal shares end at different times: the last part of each share is
        // handed out to the warps that finish first.
        if (pl.tails && a.pos_per_warp >= kTailMinPos) {
            const long long share_rows = a.pos_per_warp * (a.contiguous ? a.vpage : a.page_size);
            a.tail = int(a.pos_per_warp / (share_rows <= kShortShareRows ? kTailDivShort : kTailDiv));
            a.tail_pieces = a.tail >= kTailPieces ? kTailPieces : 1;
            a.tail_ctl = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(a.flags) + kTailCtlOff);
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block_threads(pl));
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = stream;
        void* args[] = {&a, &maps[0], &maps[1]};
        if (prof) mark(&g_prof.decode_marks, stream);
        e = cudaLaunchKernelExC(&cfg, pl.ks.variant[variant], args);
        if (prof) mark(&g_prof.decode_marks, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    } else {
        a.pos_per_warp = 1;
    }
    pd::MergeArgs m{};
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.indptr = a.indptr;
    m.o = a.o;
    m.lse = a.lse;
    m.flags = a.flags;
    m.batch = a.batch;
    m.num_qo_heads = a.num_qo_heads;
    m.num_kv_heads = pl.walk_kv;
    m.group = a.group;
    m.head_tiles = a.head_tiles;
    m.heads_per_tile = a.heads_per_tile;
    m.G = pl.G;
    m.n_pos = a.n_pos;
    m.pos_per_warp = a.pos_per_warp;
    m.tail = a.tail;
    m.tail_pieces = a.tail_pieces;
    m.contiguous = a.contiguous;
    m.npv = a.npv;
    m.append = (a.k_new != nullptr && !a.contiguous) ? 1 : 0;
    const long long pairs = pl.segments * pl.heads_per_tile;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned((pairs + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* margs[] = {&m};
    if (prof) mark(&g_prof.merge_marks, stream);
    // one wave of 4-warp blocks at 4 per SM: the wide merge (fewer round trips)
    const void* mk = pairs <= (long long)pl.sms * 16 ? pl.ks.merge_wide : pl.ks.merge;
    e = cudaLaunchKernelExC(&cfg, mk, margs);
    if (prof) mark(&g_prof.merge_marks, stream);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return ok();
}

// ---------------------------------------------------------------- append / copy kernels

// One warp per (request, kv head): copy the new K and V rows into their slot.
__global__ void __launch_bounds__(128) append_kernel(const uint8_t* k_new, const uint8_t* v_new, uint8_t* k_data,
                                                     uint8_t* v_data, const int32_t* indices, const int32_t* indptr,
                                                     const int32_t* last_page_len, int batch, int Hk, int row_bytes,
                                                     int page_size, int num_total_pages, int num_indices, int* flags) {
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (w >= (long long)batch * Hk) return;
    const int b = int(w / Hk), kh = int(w % Hk);
    const int lo = __ldg(indptr + b), hi = __ldg(indptr + b + 1);
    if (hi <= lo || lo < 0 || hi > num_indices) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadIndptr);
        return;
    }
    const int page = __ldg(indices + hi - 1);
    const int slot = __ldg(last_page_len + b) - 1;
    if (page < 0 || page >= num_total_pages) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadPage);
        return;
    }
    if (slot < 0 || slot >= page_size) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadLastPageLen);
        return;
    }
    const size_t dst = ((size_t(page) * Hk + kh) * page_size + slot) * size_t(row_bytes);
    const size_t src = (size_t(b) * Hk + kh) * size_t(row_bytes);
    for (int off = lane * 16; off < row_bytes; off += 32 * 16) {
        *reinterpret_cast<uint4*>(k_data + dst + off) = __ldg(reinterpret_cast<const uint4*>(k_new + src + off));
        *reinterpret_cast<uint4*>(v_data + dst + off) = __ldg(reinterpret_cast<const uint4*>(v_new + src + off));
    }
}

// E4M3 pool: one warp per (request, kv head) writes the codes of the new K and
// V rows into their slot (the table checks of append_kernel): code =
// E4M3(x / scale[kv head]), x widened to f32, the division in f32 (IEEE,
// rounded to nearest), the conversion rounding to nearest even and
// saturating at +-448.
template <typename T>
__global__ void __launch_bounds__(128) append_fp8_kernel(const T* k_new, const T* v_new, const float* k_scale,
                                                         const float* v_scale, uint8_t* k_data, uint8_t* v_data,
                                                         const int32_t* indices, const int32_t* indptr,
                                                         const int32_t* last_page_len, int batch, int Hk, int D,
                                                         int page_size, int num_total_pages, int num_indices,
                                                         int* flags) {
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (w >= (long long)batch * Hk) return;
    const int b = int(w / Hk), kh = int(w % Hk);
    const int lo = __ldg(indptr + b), hi = __ldg(indptr + b + 1);
    if (hi <= lo || lo < 0 || hi > num_indices) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadIndptr);
        return;
    }
    const int page = __ldg(indices + hi - 1);
    const int slot = __ldg(last_page_len + b) - 1;
    if (page < 0 || page >= num_total_pages) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadPage);
        return;
    }
    if (slot < 0 || slot >= page_size) {
        if (lane == 0 && kh == 0) atomicOr(flags, pd::kFlagBadLastPageLen);
        return;
    }
    const size_t dst = ((size_t(page) * Hk + kh) * page_size + slot) * size_t(D);
    const size_t src = (size_t(b) * Hk + kh) * size_t(D);
    const float ks = __ldg(k_scale + kh), vs = __ldg(v_scale + kh);
    for (int e = lane * 8; e < D; e += 32 * 8) {
        float fk[8], fv[8];
        pd::Elt<T>::to_f32(__ldg(reinterpret_cast<const uint4*>(k_new + src + e)), fk);
        pd::Elt<T>::to_f32(__ldg(reinterpret_cast<const uint4*>(v_new + src + e)), fv);
        uint32_t ck[2] = {0, 0}, cv[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 qk = make_float2(__fdiv_rn(fk[2 * i], ks), __fdiv_rn(fk[2 * i + 1], ks));
            const float2 qv = make_float2(__fdiv_rn(fv[2 * i], vs), __fdiv_rn(fv[2 * i + 1], vs));
            ck[i / 2] |= uint32_t(__nv_cvt_float2_to_fp8x2(qk, __NV_SATFINITE, __NV_E4M3)) << (16 * (i % 2));
            cv[i / 2] |= uint32_t(__nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3)) << (16 * (i % 2));
        }
        *reinterpret_cast<uint2*>(k_data + dst + e) = make_uint2(ck[0], ck[1]);
        *reinterpret_cast<uint2*>(v_data + dst + e) = make_uint2(cv[0], cv[1]);
    }
}

// One warp per (request, kv head): copy the new K and V rows into token
// `position` of the contiguous cache, HND [b, Hk, max_kv_len, D] or NHD
// [b, max_kv_len, Hk, D].
__global__ void __launch_bounds__(128) contiguous_append_kernel(const uint8_t* k_new, const uint8_t* v_new,
                                                                uint8_t* k_cache, uint8_t* v_cache, int batch, int Hk,
                                                                int row_bytes, long long max_kv_len, int position,
                                                                int nhd) {
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (w >= (long long)batch * Hk) return;
    const long long b = w / Hk, kh = w % Hk;
    const size_t row = nhd ? (size_t(b) * size_t(max_kv_len) + size_t(position)) * size_t(Hk) + size_t(kh)
                           : size_t(w) * size_t(max_kv_len) + size_t(position);
    const size_t dst = row * size_t(row_bytes);
    const size_t src = size_t(w) * size_t(row_bytes);
    for (int off = lane * 16; off < row_bytes; off += 32 * 16) {
        *reinterpret_cast<uint4*>(k_cache + dst + off) = __ldg(reinterpret_cast<const uint4*>(k_new + src + off));
        *reinterpret_cast<uint4*>(v_cache + dst + off) = __ldg(reinterpret_cast<const uint4*>(v_new + src + off));
    }
}

// Plain streaming copy: four independent 16-byte loads in flight per thread.
__global__ void __launch_bounds__(512) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, size_t n) {
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
                    d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

pd_status check_workspace(void* ws, size_t have, size_t need) {
    if (ws == nullptr) return fail(PD_ERR_WORKSPACE, "workspace is null (needed %zu bytes)", need);
    if (!aligned(ws, 256)) return fail(PD_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
    if (have < need) return fail(PD_ERR_WORKSPACE, "workspace too small: needed %zu bytes, got %zu", need, have);
    return PD_OK;
}

}  // namespace

extern "C" {

int pd_version(void) { return PD_VERSION; }

const char* pd_last_error_string(void) { return g_err; }

size_t pd_paged_decode_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads, int head_dim, pd_dtype dtype) {
    Plan p;
    if (make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, false, &p) != PD_OK) return 0;
    ok();
    return p.ws_bytes;
}

int pd_decode_kernel_kind(int num_qo_heads, int num_kv_heads, int head_dim, pd_dtype dtype, int fp8_pool) {
    if (num_qo_heads <= 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0) return PD_KERNEL_NONE;
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return PD_KERNEL_NONE;
    if (fp8_pool && dtype == PD_F32) return PD_KERNEL_NONE;
    // the tile rule of make_plan_uncached; the lookups only take kernel addresses
    int tiles = 0, per = 0;
    split_group(num_qo_heads / num_kv_heads, &tiles, &per);
    int G = 1;
    while (G < per) G *= 2;
    pd::KernelSet ks{};
    if (!(fp8_pool ? lookup_fp8(dtype, head_dim, G, kv_pairs_ok(dtype, num_qo_heads, num_kv_heads), &ks)
                   : lookup(dtype, head_dim, G, &ks)))
        return PD_KERNEL_NONE;
    return ks.mma == 3   ? PD_KERNEL_FP8_TCGEN05
           : ks.mma == 2 ? PD_KERNEL_FP8_TENSOR_CORES
           : ks.mma == 1 ? PD_KERNEL_TENSOR_CORES
                         : PD_KERNEL_CUDA_CORES;
}

size_t pd_contiguous_decode_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                            pd_dtype dtype) {
    Plan p;
    if (make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, true, &p) != PD_OK) return 0;
    ok();
    return p.ws_bytes;
}

// The paged decode, with the fused append when k_new / v_new are not null,
// over an E4M3 pool when k_scale / v_scale are not null.
static pd_status paged_decode_impl(const void* q, const void* k_new, const void* v_new, const void* k_data,
                                   const void* v_data, const int32_t* indices, const int32_t* indptr,
                                   const int32_t* last_page_len, void* o, float* lse, int batch, int num_qo_heads,
                                   int num_kv_heads, int head_dim, int page_size, int num_total_pages,
                                   int num_indices, float sm_scale, pd_dtype dtype, void* workspace,
                                   size_t workspace_bytes, void* stream, const float* k_scale = nullptr,
                                   const float* v_scale = nullptr, bool clear_header = false) {
    const bool fp8 = k_scale != nullptr;
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (batch <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || page_size <= 0 || num_total_pages <= 0)
        return fail(PD_ERR_INVALID, "batch, num_qo_heads, num_kv_heads, page_size and num_total_pages must be positive");
    if (num_indices < 0) return fail(PD_ERR_INVALID, "num_indices must not be negative");
    if (num_qo_heads % num_kv_heads != 0)
        return fail(PD_ERR_INVALID, "num_qo_heads (%d) must be a multiple of num_kv_heads (%d)", num_qo_heads, num_kv_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!std::isfinite(sm_scale)) return fail(PD_ERR_INVALID, "sm_scale must be finite");
    if (!q || !k_data || !v_data || !indptr || !last_page_len || !o || !lse || (num_indices > 0 && !indices))
        return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(q, 16) || !aligned(k_data, 16) || !aligned(v_data, 16) || !aligned(o, 16))
        return fail(PD_ERR_UNSUPPORTED, "q, k_data, v_data and o must be 16-byte aligned");
    if (!aligned(lse, 4) || !aligned(indptr, 4) || !aligned(last_page_len, 4) || (indices && !aligned(indices, 4)))
        return fail(PD_ERR_UNSUPPORTED, "lse, indices, indptr and last_page_len must be 4-byte aligned");
    Plan pl;
    pd_status st = make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, false, &pl, fp8);
    if (st != PD_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, pl.ws_bytes)) != PD_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    pd::DecodeArgs a{};
    a.q = q;
    a.k = k_data;
    a.v = v_data;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.indices = indices;
    a.indptr = indptr;
    a.last_page_len = last_page_len;
    a.o = o;
    a.lse = lse;
    a.part_lse = reinterpret_cast<float*>(ws + pl.lse_off);
    a.part_o = reinterpret_cast<float*>(ws + pl.o_off);
    a.flags = reinterpret_cast<int*>(ws);
    a.batch = batch;
    a.num_qo_heads = num_qo_heads;
    a.num_kv_heads = num_kv_heads;
    a.page_size = page_size;
    a.num_total_pages = num_total_pages;
    a.group = pl.group;
    a.head_tiles = pl.head_tiles;
    a.heads_per_tile = pl.heads_per_tile;
    a.n_pos = num_indices;
    a.table_bytes = pl.table_bytes;
    a.total_pos = (long long)pl.head_tiles * pl.walk_kv * num_indices;
    a.q_scale = sm_scale * pd::kLog2e;
    a.contiguous = 0;
    a.slab_rows = page_size;
    a.k_new = k_new;
    a.v_new = v_new;
    if (clear_header) {
        // Every check has passed: zero the status word and the tail counters
        // (a workspace whose header the caller cannot clear itself).
        const cudaError_t e =
            cudaMemsetAsync(workspace, 0, PD_WORKSPACE_HEADER_BYTES, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
    }
    return launch_decode(pl, a, head_dim, dtype, num_total_pages, false, static_cast<cudaStream_t>(stream));
}

pd_status pd_paged_decode(const void* q, const void* k_data, const void* v_data, const int32_t* indices,
                          const int32_t* indptr, const int32_t* last_page_len, void* o, float* lse, int batch,
                          int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int num_total_pages,
                          int num_indices, float sm_scale, pd_dtype dtype, void* workspace, size_t workspace_bytes,
                          void* stream) {
    return paged_decode_impl(q, nullptr, nullptr, k_data, v_data, indices, indptr, last_page_len, o, lse, batch,
                             num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices, sm_scale,
                             dtype, workspace, workspace_bytes, stream);
}

size_t pd_paged_decode_fp8_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                           pd_dtype dtype) {
    Plan p;
    if (make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, false, &p, true) != PD_OK) return 0;
    ok();
    return p.ws_bytes;
}

pd_status pd_paged_decode_fp8(const void* q, const void* k_data, const void* v_data, const float* k_scale,
                              const float* v_scale, const int32_t* indices, const int32_t* indptr,
                              const int32_t* last_page_len, void* o, float* lse, int batch, int num_qo_heads,
                              int num_kv_heads, int head_dim, int page_size, int num_total_pages, int num_indices,
                              float sm_scale, pd_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "E4M3 pools take PD_F16 or PD_BF16 q and o");
    if (!k_scale || !v_scale) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_scale, 4) || !aligned(v_scale, 4)) return fail(PD_ERR_UNSUPPORTED, "k_scale and v_scale must be 4-byte aligned");
    return paged_decode_impl(q, nullptr, nullptr, k_data, v_data, indices, indptr, last_page_len, o, lse, batch,
                             num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices, sm_scale,
                             dtype, workspace, workspace_bytes, stream, k_scale, v_scale);
}

pd_status pd_paged_append_decode(const void* q, const void* k_new, const void* v_new, void* k_data, void* v_data,
                                 const int32_t* indices, const int32_t* indptr, const int32_t* last_page_len, void* o,
                                 float* lse, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                 int page_size, int num_total_pages, int num_indices, float sm_scale, pd_dtype dtype,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_new || !v_new) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(PD_ERR_UNSUPPORTED, "k_new and v_new must be 16-byte aligned");
    return paged_decode_impl(q, k_new, v_new, k_data, v_data, indices, indptr, last_page_len, o, lse, batch,
                             num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices, sm_scale,
                             dtype, workspace, workspace_bytes, stream);
}

// The contiguous decode, with the fused append of row valid_kv_len - 1 when
// k_new / v_new are not null; nhd: the cache is [batch, max_kv_len, Hk, D].
static pd_status contiguous_decode_impl(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                                        const void* v_cache, void* o, float* lse, int batch, int num_qo_heads,
                                        int num_kv_heads, int head_dim, int max_kv_len, int valid_kv_len,
                                        float sm_scale, pd_dtype dtype, void* workspace, size_t workspace_bytes,
                                        bool nhd, void* stream) {
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (batch <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || max_kv_len <= 0)
        return fail(PD_ERR_INVALID, "batch, num_qo_heads, num_kv_heads and max_kv_len must be positive");
    if (valid_kv_len < 0 || valid_kv_len > max_kv_len)
        return fail(PD_ERR_INVALID, "valid_kv_len (%d) must be in [0, max_kv_len=%d]", valid_kv_len, max_kv_len);
    if (num_qo_heads % num_kv_heads != 0)
        return fail(PD_ERR_INVALID, "num_qo_heads (%d) must be a multiple of num_kv_heads (%d)", num_qo_heads, num_kv_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!std::isfinite(sm_scale)) return fail(PD_ERR_INVALID, "sm_scale must be finite");
    if (!q || !k_cache || !v_cache || !o) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16))
        return fail(PD_ERR_UNSUPPORTED, "q, k_cache, v_cache and o must be 16-byte aligned");
    if (lse && !aligned(lse, 4)) return fail(PD_ERR_UNSUPPORTED, "lse must be 4-byte aligned");
    Plan pl;
    pd_status st = make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, true, &pl);
    if (st != PD_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, pl.ws_bytes)) != PD_OK) return st;
    const int vpage = 4 * pl.ks.rows_per_stage;  // rows per work position
    const int npv = (valid_kv_len + vpage - 1) / vpage;
    const long long n_pos = (long long)batch * npv;
    if (n_pos > 0x7fffffffLL) return fail(PD_ERR_UNSUPPORTED, "batch * max_kv_len too large");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    pd::DecodeArgs a{};
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.o = o;
    a.lse = lse;
    a.part_lse = reinterpret_cast<float*>(ws + pl.lse_off);
    a.part_o = reinterpret_cast<float*>(ws + pl.o_off);
    a.flags = reinterpret_cast<int*>(ws);
    a.batch = batch;
    a.num_qo_heads = num_qo_heads;
    a.num_kv_heads = num_kv_heads;
    a.page_size = vpage;
    a.num_total_pages = 1;
    a.group = pl.group;
    a.head_tiles = pl.head_tiles;
    a.heads_per_tile = pl.heads_per_tile;
    a.n_pos = int(n_pos);
    a.table_bytes = 0;
    a.total_pos = (long long)pl.head_tiles * num_kv_heads * n_pos;
    a.q_scale = sm_scale * pd::kLog2e;
    a.contiguous = 1;
    a.slab_rows = max_kv_len;
    a.valid_kv_len = valid_kv_len;
    a.vpage = vpage;
    a.npv = npv;
    a.k_new = k_new;
    a.v_new = v_new;
    return launch_decode(pl, a, head_dim, dtype, batch, nhd, static_cast<cudaStream_t>(stream));
}

pd_status pd_contiguous_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                               int batch, int num_qo_heads, int num_kv_heads, int head_dim, int max_kv_len,
                               int valid_kv_len, float sm_scale, pd_dtype dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return contiguous_decode_impl(q, nullptr, nullptr, k_cache, v_cache, o, lse, batch, num_qo_heads, num_kv_heads,
                                  head_dim, max_kv_len, valid_kv_len, sm_scale, dtype, workspace, workspace_bytes,
                                  false, stream);
}

pd_status pd_contiguous_append_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                      void* v_cache, void* o, float* lse, int batch, int num_qo_heads,
                                      int num_kv_heads, int head_dim, int max_kv_len, int position, float sm_scale,
                                      pd_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_new || !v_new) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(PD_ERR_UNSUPPORTED, "k_new and v_new must be 16-byte aligned");
    if (position < 0 || position >= max_kv_len)
        return fail(PD_ERR_INVALID, "position (%d) must be in [0, max_kv_len=%d)", position, max_kv_len);
    return contiguous_decode_impl(q, k_new, v_new, k_cache, v_cache, o, lse, batch, num_qo_heads, num_kv_heads,
                                  head_dim, max_kv_len, position + 1, sm_scale, dtype, workspace, workspace_bytes,
                                  false, stream);
}

pd_status pd_contiguous_decode_nhd(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                               int batch, int num_qo_heads, int num_kv_heads, int head_dim, int max_kv_len,
                               int valid_kv_len, float sm_scale, pd_dtype dtype, void* workspace,
                               size_t workspace_bytes, void* stream) {
    return contiguous_decode_impl(q, nullptr, nullptr, k_cache, v_cache, o, lse, batch, num_qo_heads, num_kv_heads,
                                  head_dim, max_kv_len, valid_kv_len, sm_scale, dtype, workspace, workspace_bytes,
                                  true, stream);
}

pd_status pd_contiguous_append_decode_nhd(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                      void* v_cache, void* o, float* lse, int batch, int num_qo_heads,
                                      int num_kv_heads, int head_dim, int max_kv_len, int position, float sm_scale,
                                      pd_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (!k_new || !v_new) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(PD_ERR_UNSUPPORTED, "k_new and v_new must be 16-byte aligned");
    if (position < 0 || position >= max_kv_len)
        return fail(PD_ERR_INVALID, "position (%d) must be in [0, max_kv_len=%d)", position, max_kv_len);
    return contiguous_decode_impl(q, k_new, v_new, k_cache, v_cache, o, lse, batch, num_qo_heads, num_kv_heads,
                                  head_dim, max_kv_len, position + 1, sm_scale, dtype, workspace, workspace_bytes,
                                  true, stream);
}


pd_status pd_paged_append(const void* k_new, const void* v_new, void* k_data, void* v_data, const int32_t* indices,
                          const int32_t* indptr, const int32_t* last_page_len, int batch, int num_kv_heads,
                          int head_dim, int page_size, int num_total_pages, int num_indices, pd_dtype dtype,
                          void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (batch <= 0 || num_kv_heads <= 0 || page_size <= 0 || num_total_pages <= 0 || num_indices < 0)
        return fail(PD_ERR_INVALID, "batch, num_kv_heads, page_size and num_total_pages must be positive");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!k_new || !v_new || !k_data || !v_data || !indptr || !last_page_len || (num_indices > 0 && !indices))
        return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_data, 16) || !aligned(v_data, 16))
        return fail(PD_ERR_UNSUPPORTED, "k_new, v_new, k_data and v_data must be 16-byte aligned");
    pd_status st = check_workspace(workspace, workspace_bytes, PD_WORKSPACE_HEADER_BYTES);
    if (st != PD_OK) return st;
    const long long warps = (long long)batch * num_kv_heads;
    std::unique_lock<std::mutex> plk(g_prof_mu);
    const bool prof = g_prof.on;
    if (!prof) plk.unlock();
    if (prof) mark(&g_prof.append_marks, static_cast<cudaStream_t>(stream));
    append_kernel<<<unsigned((warps + 3) / 4), 128, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new), static_cast<uint8_t*>(k_data),
        static_cast<uint8_t*>(v_data), indices, indptr, last_page_len, batch, num_kv_heads,
        int(head_dim * elem_size(dtype)), page_size, num_total_pages, num_indices, static_cast<int*>(workspace));
    cudaError_t e = cudaGetLastError();
    if (prof) mark(&g_prof.append_marks, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return ok();
}

static pd_status contiguous_append_impl(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                        int batch, int num_kv_heads, int head_dim, int max_kv_len, int position,
                                        pd_dtype dtype, bool nhd, void* stream) {
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (batch <= 0 || num_kv_heads <= 0 || max_kv_len <= 0)
        return fail(PD_ERR_INVALID, "batch, num_kv_heads and max_kv_len must be positive");
    if (position < 0 || position >= max_kv_len)
        return fail(PD_ERR_INVALID, "position (%d) must be in [0, max_kv_len=%d)", position, max_kv_len);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!k_new || !v_new || !k_cache || !v_cache) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return fail(PD_ERR_UNSUPPORTED, "k_new, v_new, k_cache and v_cache must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::unique_lock<std::mutex> plk(g_prof_mu);
    const bool prof = g_prof.on;
    if (!prof) plk.unlock();
    if (prof) mark(&g_prof.append_marks, s);
    const long long warps = (long long)batch * num_kv_heads;
    contiguous_append_kernel<<<unsigned((warps + 3) / 4), 128, 0, s>>>(
        static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new), static_cast<uint8_t*>(k_cache),
        static_cast<uint8_t*>(v_cache), batch, num_kv_heads, int(head_dim * elem_size(dtype)), max_kv_len, position, nhd ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (prof) mark(&g_prof.append_marks, s);
    if (e != cudaSuccess) return cuda_fail(e, "contiguous append launch");
    return ok();
}

pd_status pd_paged_append_fp8(const void* k_new, const void* v_new, const float* k_scale, const float* v_scale,
                              void* k_data, void* v_data, const int32_t* indices, const int32_t* indptr,
                              const int32_t* last_page_len, int batch, int num_kv_heads, int head_dim, int page_size,
                              int num_total_pages, int num_indices, pd_dtype dtype, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "k_new and v_new must be PD_F16 or PD_BF16");
    if (batch <= 0 || num_kv_heads <= 0 || page_size <= 0 || num_total_pages <= 0 || num_indices < 0)
        return fail(PD_ERR_INVALID, "batch, num_kv_heads, page_size and num_total_pages must be positive");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!k_new || !v_new || !k_scale || !v_scale || !k_data || !v_data || !indptr || !last_page_len ||
        (num_indices > 0 && !indices))
        return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_data, 16) || !aligned(v_data, 16) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return fail(PD_ERR_UNSUPPORTED, "k_new, v_new, k_data, v_data must be 16-byte and the scales 4-byte aligned");
    pd_status st = check_workspace(workspace, workspace_bytes, PD_WORKSPACE_HEADER_BYTES);
    if (st != PD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long warps = (long long)batch * num_kv_heads;
    std::unique_lock<std::mutex> plk(g_prof_mu);
    const bool prof = g_prof.on;
    if (!prof) plk.unlock();
    if (prof) mark(&g_prof.append_marks, s);
    const unsigned grid = unsigned((warps + 3) / 4);
    if (dtype == PD_F16)
        append_fp8_kernel<__half><<<grid, 128, 0, s>>>(
            static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), k_scale, v_scale,
            static_cast<uint8_t*>(k_data), static_cast<uint8_t*>(v_data), indices, indptr, last_page_len, batch,
            num_kv_heads, head_dim, page_size, num_total_pages, num_indices, static_cast<int*>(workspace));
    else
        append_fp8_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
            static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), k_scale, v_scale,
            static_cast<uint8_t*>(k_data), static_cast<uint8_t*>(v_data), indices, indptr, last_page_len, batch,
            num_kv_heads, head_dim, page_size, num_total_pages, num_indices, static_cast<int*>(workspace));
    cudaError_t e = cudaGetLastError();
    if (prof) mark(&g_prof.append_marks, s);
    if (e != cudaSuccess) return cuda_fail(e, "fp8 append launch");
    return ok();
}

pd_status pd_contiguous_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int batch,
                               int num_kv_heads, int head_dim, int max_kv_len, int position, pd_dtype dtype,
                               void* stream) {
    return contiguous_append_impl(k_new, v_new, k_cache, v_cache, batch, num_kv_heads, head_dim, max_kv_len, position,
                                  dtype, false, stream);
}

pd_status pd_contiguous_append_nhd(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int batch,
                                   int num_kv_heads, int head_dim, int max_kv_len, int position, pd_dtype dtype,
                                   void* stream) {
    return contiguous_append_impl(k_new, v_new, k_cache, v_cache, batch, num_kv_heads, head_dim, max_kv_len, position,
                                  dtype, true, stream);
}

pd_status pd_merge_states(const float* o_parts, const float* lse_parts, int num_parts, int num_rows, int head_dim,
                          void* o, float* lse, pd_dtype dtype, void* stream) {
    if (dtype != PD_F32 && dtype != PD_F16 && dtype != PD_BF16) return fail(PD_ERR_UNSUPPORTED, "dtype must be PD_F32, PD_F16 or PD_BF16");
    if (num_parts <= 0 || num_rows < 0) return fail(PD_ERR_INVALID, "num_parts must be positive and num_rows not negative");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PD_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    if (!o_parts || !lse_parts || !o) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(o_parts, 16) || !aligned(o, 16)) return fail(PD_ERR_UNSUPPORTED, "o_parts and o must be 16-byte aligned");
    if (num_rows == 0) return ok();
    pd::KernelSet ks{};
    if (!lookup(dtype, head_dim, 1, &ks)) return fail(PD_ERR_UNSUPPORTED, "no merge kernel for this head_dim");
    const void* fn = ks.merge_states;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned((num_rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    void* args[] = {&o_parts, &lse_parts, &num_parts, &num_rows, &o, &lse};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return cuda_fail(e, "merge_states launch");
    return ok();
}

pd_status pd_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    pd_status st = check_workspace(workspace, workspace_bytes, PD_WORKSPACE_HEADER_BYTES);
    if (st != PD_OK) return st;
    cudaError_t e = cudaMemsetAsync(workspace, 0, PD_WORKSPACE_HEADER_BYTES, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    return ok();
}

pd_status pd_read_device_flags(const void* workspace, int32_t* flags, void* stream) {
    if (!workspace || !flags) return fail(PD_ERR_INVALID, "null pointer argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(flags, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    return ok();
}

pd_status pd_copy_bytes(void* dst, const void* src, size_t bytes, void* stream) {
    if (!dst || !src) return fail(PD_ERR_INVALID, "null pointer argument");
    if (!aligned(dst, 16) || !aligned(src, 16) || bytes % 16 != 0)
        return fail(PD_ERR_UNSUPPORTED, "dst, src and bytes must be multiples of 16");
    if (bytes == 0) return ok();
    DeviceInfo di;
    pd_status st = device_info(&di);
    if (st != PD_OK) return st;
    copy_kernel<<<di.sms * 4, 512, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(dst), static_cast<const uint4*>(src), bytes / 16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "copy launch");
    return ok();
}

pd_status pd_select_fp8_kernel(int kind) {
    if (kind != PD_KERNEL_FP8_TENSOR_CORES && kind != PD_KERNEL_FP8_TCGEN05)
        return fail(PD_ERR_INVALID, "kind must be PD_KERNEL_FP8_TENSOR_CORES or PD_KERNEL_FP8_TCGEN05");
    g_fp8_tcgen05.store(kind == PD_KERNEL_FP8_TCGEN05 ? 1 : 0, std::memory_order_relaxed);
    return ok();
}

pd_status pd_test_inject_wait_timeout(int extra_bytes) {
    if (extra_bytes < 0 || extra_bytes > (1 << 20) || extra_bytes % 16 != 0)
        return fail(PD_ERR_INVALID, "extra_bytes must be a multiple of 16 in [0, 1 MiB]");
    g_inject_extra_tx.store(extra_bytes, std::memory_order_relaxed);
    return ok();
}

pd_status pd_profile_enable(int enable) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.on = enable != 0;
    return ok();
}

pd_status pd_profile_read(double* decode_ms, int* decode_launches, double* merge_ms, int* merge_launches,
                          double* append_ms, int* append_launches) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    auto sum = [](std::vector<cudaEvent_t>& v, double* ms, int* n) -> cudaError_t {
        double t = 0;
        int cnt = 0;
        cudaError_t err = cudaSuccess;
        for (size_t i = 0; i + 1 < v.size(); i += 2) {
            float x = 0;
            err = cudaEventSynchronize(v[i + 1]);
            if (err == cudaSuccess) err = cudaEventElapsedTime(&x, v[i], v[i + 1]);
            if (err != cudaSuccess) break;
            t += x;
            ++cnt;
        }
        for (cudaEvent_t e : v) g_prof.free_events.push_back(e);
        v.clear();
        if (ms) *ms = t;
        if (n) *n = cnt;
        return err;
    };
    cudaError_t e1 = sum(g_prof.decode_marks, decode_ms, decode_launches);
    cudaError_t e2 = sum(g_prof.merge_marks, merge_ms, merge_launches);
    cudaError_t e3 = sum(g_prof.append_marks, append_ms, append_launches);
    if (e1 != cudaSuccess) return cuda_fail(e1, "reading decode events");
    if (e2 != cudaSuccess) return cuda_fail(e2, "reading merge events");
    if (e3 != cudaSuccess) return cuda_fail(e3, "reading append events");
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------- decode with built-in scratch
//
// Some callers cannot allocate device memory when they call the decode: an
// engine plugin whose host framework owns every device buffer and hands the
// op no scratch, or a serving loop that bans cudaMalloc on its hot path
// because it can synchronize the device and fragment the memory pool. For
// them pd_paged_decode_noalloc runs the same decode with its scratch in the
// fixed-size array below, which every device that loads this library keeps
// for the life of the process.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
std::vector<void*> g_noalloc_addr;  // device address of the array, per device ordinal

// The host-side name of a __device__ array is not its device address; ask the
// runtime for it once per device, with that device current.
pd_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (int(g_noalloc_addr.size()) <= dev) g_noalloc_addr.resize(dev + 1, nullptr);
    if (g_noalloc_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode scratch)");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return PD_OK;
}

}  // namespace

extern "C" pd_status pd_paged_decode_noalloc(const void* q, const void* k_data, const void* v_data,
                                             const int32_t* indices, const int32_t* indptr,
                                             const int32_t* last_page_len, void* o, float* lse, int batch,
                                             int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                                             int num_total_pages, int num_indices, float sm_scale, pd_dtype dtype,
                                             void* stream) {
    void* scratch = nullptr;
    pd_status st = noalloc_scratch(&scratch);
    if (st != PD_OK) return st;
    Plan pl;
    if ((st = make_plan(dtype, batch, num_qo_heads, num_kv_heads, head_dim, false, &pl)) != PD_OK) return st;
    if (pl.ws_bytes > kNoAllocScratchBytes)
        return fail(PD_ERR_WORKSPACE,
                    "this shape needs %zu bytes of decode scratch; pd_paged_decode_noalloc has %zu "
                    "(use pd_paged_decode with a caller workspace)",
                    pl.ws_bytes, kNoAllocScratchBytes);
    // The array keeps the last call's contents: its header (status word and
    // tail counters) is cleared once every argument check has passed, just
    // before the launch, so a rejected call enqueues nothing.
    return paged_decode_impl(q, nullptr, nullptr, k_data, v_data, indices, indptr, last_page_len, o, lse, batch,
                             num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices, sm_scale,
                             dtype, scratch, kNoAllocScratchBytes, stream, nullptr, nullptr, true);
}

extern "C" pd_status pd_paged_decode_noalloc_flags(int32_t* flags, void* stream) {
    if (!flags) return fail(PD_ERR_INVALID, "null pointer argument");
    void* scratch = nullptr;
    pd_status st = noalloc_scratch(&scratch);
    if (st != PD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(flags, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the static scratch status word");
    return ok();
}
