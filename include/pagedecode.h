/*
 * pagedecode: batched single-query (decode-phase) grouped-query attention over
 * a paged KV cache, for NVIDIA sm_103a (GB300).
 *
 * The problem statement followed here is the module documentation of
 * baracuda-kernels 0.0.1-alpha.68, src/attention/batch_paged_decode.rs,
 * sections "Layout" and "Constraints", and its descriptor and argument types
 * (PagedKvCacheDescriptor, BatchPagedDecodeDescriptor, BatchPagedDecodeArgs):
 *
 *   k_data, v_data  [num_total_pages, num_kv_heads, page_size, head_dim]  T, HND
 *   indices         [num_indices]  int32  physical page ids
 *   indptr          [batch + 1]    int32  request b owns indices[indptr[b] .. indptr[b+1])
 *   last_page_len   [batch]        int32  valid rows in request b's last page, 0..page_size
 *   q, o            [batch, num_qo_heads, head_dim]  T
 *   lse             [batch, num_qo_heads]  float32 (whatever T is)
 *
 * For request b with np = indptr[b+1] - indptr[b] pages, kv_len = (np - 1) *
 * page_size + last_page_len[b] (0 when np = 0); token t is row t % page_size of
 * page indices[indptr[b] + t / page_size]. Query head h reads kv head
 * h / (num_qo_heads / num_kv_heads) (ferrox-cuda 0.15.2, src/attn.rs,
 * gqa_decode). With s_t = sm_scale * q[b,h,:] . k_t:
 *
 *   o[b,h,:]  = sum_t exp(s_t - lse) * v_t        lse[b,h] = ln sum_t exp(s_t)
 *
 * An empty request (kv_len = 0) gets o = 0 and lse = -infinity.
 *
 * Conventions shared by every call:
 *  - Pointers marked "device" are CUDA device pointers (or managed memory) on
 *    the current device; host pointers are marked "host". The caller owns
 *    every buffer, including the page table and its allocator; the library
 *    allocates no memory on any call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream). No call blocks the host except the two marked "synchronizes".
 *  - T is given by `dtype`: PD_F32 float, PD_F16 IEEE half, PD_BF16 bfloat16.
 *    Accumulation is float32 for every T. Results are bit-identical across
 *    repeated calls with the same arguments on the same device.
 *  - Arguments are checked on the host before anything is enqueued; a failed
 *    check returns an error status, enqueues nothing and sets the message
 *    returned by pd_last_error_string(). Values that live in device memory
 *    (page ids, indptr, last_page_len) are checked by the kernels: a bad
 *    value sets a bit of the sticky status word in the workspace header (see
 *    PD_FLAG_*), the offending page or request is treated as empty, and the
 *    kernel carries on. No kernel traps. A malformed indptr (decreasing,
 *    negative or past num_indices: PD_FLAG_BAD_INDPTR) makes request ranges
 *    overlap or run off the table, so it leaves every output of that call
 *    undefined, not only the flagged request's; the kernels still finish,
 *    and later calls with a good table are unaffected.
 *  - Status codes: PD_ERR_INVALID for malformed extents or null pointers,
 *    PD_ERR_UNSUPPORTED for a head_dim, dtype or pointer alignment this
 *    library does not handle, PD_ERR_WORKSPACE for a missing or small
 *    workspace, PD_ERR_CUDA when the CUDA runtime reports an error.
 */
#ifndef PAGEDECODE_H
#define PAGEDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PD_VERSION 1

typedef enum { PD_F32 = 0, PD_F16 = 1, PD_BF16 = 2 } pd_dtype;

typedef enum {
    PD_OK = 0,
    PD_ERR_INVALID = 1,
    PD_ERR_UNSUPPORTED = 2,
    PD_ERR_WORKSPACE = 3,
    PD_ERR_CUDA = 4
} pd_status;

/* Bits of the sticky device status word (first int32 of every workspace). */
#define PD_FLAG_BAD_PAGE_ID 0x1       /* a page id outside [0, num_total_pages): page treated as empty */
#define PD_FLAG_BAD_LAST_PAGE_LEN 0x2 /* last_page_len outside [0, page_size]: clamped to that range */
#define PD_FLAG_BAD_INDPTR 0x4        /* indptr decreasing, negative or past num_indices: all outputs invalid */
#define PD_FLAG_WAIT_TIMEOUT 0x8      /* a copy pipeline wait passed its time limit; outputs invalid */

/* Bytes at the start of every workspace that hold the status word and the
 * decode's work-distribution counters (zero between calls). */
#define PD_WORKSPACE_HEADER_BYTES 256

/*
 * Workspace bytes pd_paged_decode needs for this shape on the current device
 * (the split-KV partial results and the status word). Depends on the
 * device's SM count, so query it on the device that will run the call.
 * Returns 0 on a bad shape or when no device is present (see
 * pd_last_error_string()).
 */
size_t pd_paged_decode_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                       pd_dtype dtype);

/*
 * Which decode kernel a call of this shape runs: one of PD_KERNEL_*. With
 * fp8_pool nonzero the question is about pd_paged_decode_fp8 (dtype is then
 * the type of q and o); otherwise about pd_paged_decode and the contiguous
 * calls, which share their kernels. The group g = num_qo_heads / num_kv_heads
 * is served in tiles of at most 8 q heads, padded to 1, 2, 4 or 8. 16-bit
 * tiles of 4 or 8 run on tensor cores; f32 and 16-bit tiles of 1 or 2 run on
 * CUDA cores. Over E4M3 pools, tiles of 4 or 8 at head_dim 128 or 256 run on
 * the mma.sync E4M3 tensor-core kernel, or, when pd_select_fp8_kernel chose
 * it and the shape allows it (bf16 q, groups of exactly 4 q heads, an even
 * number of kv heads, head_dim 128), on the tcgen05 kernel; the rest run on
 * CUDA cores. This is a host-side
 * lookup: it needs no device, enqueues nothing and returns PD_KERNEL_NONE for
 * a shape that no call accepts.
 */
#define PD_KERNEL_NONE 0
#define PD_KERNEL_CUDA_CORES 1
#define PD_KERNEL_TENSOR_CORES 2
#define PD_KERNEL_FP8_TENSOR_CORES 3
#define PD_KERNEL_FP8_TCGEN05 4
int pd_decode_kernel_kind(int num_qo_heads, int num_kv_heads, int head_dim, pd_dtype dtype, int fp8_pool);

/*
 * Which tensor-core kernel decodes over E4M3 pools where both apply (bf16 q,
 * groups of exactly 4 q heads, an even number of kv heads, head_dim 128):
 * PD_KERNEL_FP8_TENSOR_CORES (mma.sync over codes widened in registers; the
 * default, and the faster on the measured shapes) or PD_KERNEL_FP8_TCGEN05
 * (tcgen05.mma on the codes in shared memory, accumulators in tensor memory).
 * Both give results within the same tolerances. Process-wide; it applies to
 * the calls made after it returns, and to pd_decode_kernel_kind and the
 * workspace sizes (which may differ between the two). PD_ERR_INVALID for any
 * other value.
 */
pd_status pd_select_fp8_kernel(int kind);

/*
 * Batched paged decode (batch_paged_decode.rs: BatchPagedDecodePlan::run and
 * the per-dtype FFI launch it makes, whose argument order this follows).
 *
 * q, k_data, v_data, o: device, 16-byte aligned, layouts above. o (and lse)
 *   may also be pinned host memory (cudaHostAlloc / cudaMallocHost), which
 *   kernels reach at its host address under unified addressing: the kernels
 *   then store the results straight into host memory, with no copy back.
 * indices (may be NULL only if num_indices == 0), indptr, last_page_len: device int32.
 * lse: device float32 [batch, num_qo_heads], natural log.
 * head_dim: 64, 128 or 256. num_qo_heads % num_kv_heads == 0.
 * num_total_pages: pages in k_data/v_data. num_indices: entries in indices
 *   (the host-side length of the array; indptr[batch] must not exceed it).
 * sm_scale: the score scale, used as given (typically 1/sqrt(head_dim)).
 * workspace: device, 256-byte aligned, at least
 *   pd_paged_decode_workspace_bytes(...) bytes, its header zeroed once by
 *   pd_workspace_init() before first use. Calls that share a workspace must
 *   be ordered on one stream.
 *
 * Long requests are split across warps in a load-balanced partition of all
 * (kv head, page) work; the last part of each warp's share (a quarter of
 * shares of up to 1,024 K/V rows, an eighth of longer ones) goes, at fixed
 * boundaries, to whichever warp finishes first (counters in the workspace
 * header, back at zero after every call). Partial (o, lse) pairs are combined
 * by a merge kernel in a fixed order, so results do not depend on timing.
 */
pd_status pd_paged_decode(const void* q, const void* k_data, const void* v_data,
                          const int32_t* indices, const int32_t* indptr,
                          const int32_t* last_page_len, void* o, float* lse, int batch,
                          int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                          int num_total_pages, int num_indices, float sm_scale, pd_dtype dtype,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Paged append (batch_paged_decode.rs, module doc "Companion plans":
 * PagedKvAppendPlan writes the new K/V slices into the paged store at decode
 * time; the caller owns the page table and its allocator).
 *
 * The caller first updates the page table for the new token: if request b's
 * last page is full (or it has no page) it appends a free page to its list
 * and sets last_page_len[b] = 1, otherwise it adds 1 to last_page_len[b].
 * This call then copies, bit for bit, k_new[b, h, :] and v_new[b, h, :] into
 * row last_page_len[b] - 1 of page indices[indptr[b+1] - 1], kv head h.
 *
 * k_new, v_new: device [batch, num_kv_heads, head_dim] T, 16-byte aligned.
 * k_data, v_data: device, modified in place. indices/indptr/last_page_len:
 *   device int32, the table after the caller's update.
 * workspace: device, at least PD_WORKSPACE_HEADER_BYTES bytes (the status
 *   word); a decode workspace may be shared.
 * A request with no page, a page id out of range or a last_page_len outside
 * [1, page_size] is skipped and flagged.
 */
pd_status pd_paged_append(const void* k_new, const void* v_new, void* k_data, void* v_data,
                          const int32_t* indices, const int32_t* indptr,
                          const int32_t* last_page_len, int batch, int num_kv_heads, int head_dim,
                          int page_size, int num_total_pages, int num_indices, pd_dtype dtype,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 KV pools. This is an extension of this library, not a layout of the
 * pages above: K and V pages hold one-byte E4M3 codes, in the same HND layout
 * as pd_paged_decode ([max_num_pages, num_kv_heads, page_size, head_dim]), and
 * element value = E4M3 value of the code * k_scale[h] (v_scale[h] for V), h
 * its kv head. E4M3 is the format of the OCP 8-bit floating point
 * specification (bias 7, 3 mantissa bits, S.1111.111 NaN, largest finite 448).
 * The pool is half the bytes of an f16 pool, and this decode is bound by
 * those bytes.
 *
 * pd_paged_decode_fp8: the arguments of pd_paged_decode plus k_scale, v_scale
 *   (device f32 [num_kv_heads], 4-byte aligned); dtype (PD_F16 or PD_BF16) is
 *   the type of q and o. The workspace size comes from
 *   pd_paged_decode_fp8_workspace_bytes (the stage geometry differs from the
 *   16-bit pools). Results, lse and errors as pd_paged_decode.
 * pd_paged_append_fp8: the slot of pd_paged_append receives, for each element
 *   x of k_new (v_new), the code of x / k_scale[h] (v_scale[h]): x widened to
 *   f32, the division in f32, rounded to the nearest code with ties to even,
 *   saturating at +-448 (NaN stays NaN). dtype is the type of k_new / v_new
 *   (PD_F16 or PD_BF16). Table errors as pd_paged_append.
 */
size_t pd_paged_decode_fp8_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                           pd_dtype dtype);
pd_status pd_paged_decode_fp8(const void* q, const void* k_data, const void* v_data, const float* k_scale,
                              const float* v_scale, const int32_t* indices, const int32_t* indptr,
                              const int32_t* last_page_len, void* o, float* lse, int batch,
                              int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                              int num_total_pages, int num_indices, float sm_scale, pd_dtype dtype,
                              void* workspace, size_t workspace_bytes, void* stream);
pd_status pd_paged_append_fp8(const void* k_new, const void* v_new, const float* k_scale,
                              const float* v_scale, void* k_data, void* v_data, const int32_t* indices,
                              const int32_t* indptr, const int32_t* last_page_len, int batch,
                              int num_kv_heads, int head_dim, int page_size, int num_total_pages,
                              int num_indices, pd_dtype dtype, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Append, then decode, in one kernel launch. The companion plans of
 * batch_paged_decode.rs (module doc "Companion plans": PagedKvAppendPlan, then
 * BatchPagedDecodePlan) run as two plans per decode step; this call gives
 * exactly the result of pd_paged_append followed by pd_paged_decode on the
 * same arguments. That is, the K/V pool after the call is bit for bit the one
 * pd_paged_append leaves, and o / lse are those pd_paged_decode returns on it.
 *
 * Each decode warp whose chunk holds a request's new row (row
 * last_page_len[b] - 1 of its last page) first stores that row, then reads
 * the chunk. No other launch is made for the append, and no grid-wide barrier
 * is taken.
 *
 * Arguments are those of pd_paged_decode plus k_new, v_new (device
 * [batch, num_kv_heads, head_dim] T, 16-byte aligned); k_data and v_data are
 * modified in place, and the table must already describe the new token (as for
 * pd_paged_append). A request with no page, a bad last page id or a
 * last_page_len outside [1, page_size] is not appended to and is flagged in
 * the status word; the decode of the other requests is unaffected.
 */
pd_status pd_paged_append_decode(const void* q, const void* k_new, const void* v_new, void* k_data,
                                 void* v_data, const int32_t* indices, const int32_t* indptr,
                                 const int32_t* last_page_len, void* o, float* lse, int batch,
                                 int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                                 int num_total_pages, int num_indices, float sm_scale, pd_dtype dtype,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Append to a contiguous cache (batch_paged_decode.rs, module doc "Companion
 * plans": KvCacheAppendPlan, the append to a rank-4 cache with no page
 * table). For every request b and kv head h, row `position` of
 * k_cache[b, h, :, :] becomes k_new[b, h, :], bit for bit; the same for v.
 * With the cache holding `position` valid rows before the call, a decode
 * with valid_kv_len = position + 1 then sees the new token last.
 *
 * k_new, v_new: device [batch, num_kv_heads, head_dim] T, 16-byte aligned.
 * k_cache, v_cache: device [batch, num_kv_heads, max_kv_len, head_dim] T,
 *   modified in place. 0 <= position < max_kv_len (PD_ERR_INVALID otherwise).
 */
pd_status pd_contiguous_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int batch,
                               int num_kv_heads, int head_dim, int max_kv_len, int position, pd_dtype dtype,
                               void* stream);

/*
 * pd_contiguous_append at `position`, then pd_contiguous_decode with
 * valid_kv_len = position + 1, in one launch (the contiguous-cache form of
 * pd_paged_append_decode). 0 <= position < max_kv_len (PD_ERR_INVALID
 * otherwise); k_cache, v_cache are modified in place; the workspace is that of
 * pd_contiguous_decode.
 */
pd_status pd_contiguous_append_decode(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                      void* v_cache, void* o, float* lse, int batch, int num_qo_heads,
                                      int num_kv_heads, int head_dim, int max_kv_len, int position,
                                      float sm_scale, pd_dtype dtype, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * The token-major (NHD) contiguous cache. ferrox-cuda 0.15.2, src/attn.rs
 * (gqa_decode) stores one sequence as [seq_len, n_kv_heads, head_dim]: token t
 * of kv head h starts at element (t * n_kv_heads + h) * head_dim. These three
 * calls take that layout with a batch dimension in front,
 * k_cache / v_cache [batch, max_kv_len, num_kv_heads, head_dim], and are
 * otherwise the calls of the same name without _nhd: the same arguments,
 * results, workspace (pd_contiguous_decode_workspace_bytes) and errors.
 */
pd_status pd_contiguous_decode_nhd(const void* q, const void* k_cache, const void* v_cache, void* o,
                                   float* lse, int batch, int num_qo_heads, int num_kv_heads,
                                   int head_dim, int max_kv_len, int valid_kv_len, float sm_scale,
                                   pd_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);
pd_status pd_contiguous_append_nhd(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                   int batch, int num_kv_heads, int head_dim, int max_kv_len,
                                   int position, pd_dtype dtype, void* stream);
pd_status pd_contiguous_append_decode_nhd(const void* q, const void* k_new, const void* v_new,
                                          void* k_cache, void* v_cache, void* o, float* lse, int batch,
                                          int num_qo_heads, int num_kv_heads, int head_dim,
                                          int max_kv_len, int position, float sm_scale, pd_dtype dtype,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes pd_contiguous_decode needs (same rules as above). */
size_t pd_contiguous_decode_workspace_bytes(int batch, int num_qo_heads, int num_kv_heads,
                                            int head_dim, pd_dtype dtype);

/*
 * Decode over a contiguous cache (ferrum-kernels 0.7.7,
 * src/backend/cuda/decode_attention.rs, decode_attention: q [num_q_heads,
 * head_dim], k_cache/v_cache [num_kv_heads, max_kv_len, head_dim], rows
 * [0, valid_kv_len) valid, scale), with a leading batch dimension:
 *
 * q, o: device [batch, num_qo_heads, head_dim] T, 16-byte aligned.
 * k_cache, v_cache: device [batch, num_kv_heads, max_kv_len, head_dim] T.
 * lse: device float32 [batch, num_qo_heads] or NULL to skip it.
 * 0 <= valid_kv_len <= max_kv_len; valid_kv_len = 0 gives o = 0, lse = -inf.
 * The same kernels as pd_paged_decode run with each request's rows taken as
 * consecutive pages of one contiguous block.
 */
pd_status pd_contiguous_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, int batch, int num_qo_heads, int num_kv_heads,
                               int head_dim, int max_kv_len, int valid_kv_len, float sm_scale,
                               pd_dtype dtype, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Merge attention states computed over disjoint key sets of the same query
 * rows into the state over their union: lse = ln sum_c exp(lse_c),
 * o = sum_c exp(lse_c - lse) * o_c, parts taken in index order. This is the
 * combine step of the split-KV mode, exposed so that callers holding partial
 * results from elsewhere (another device, another cache tier) can use it.
 *
 * o_parts: device float32 [num_parts, num_rows, head_dim] (each part already
 *   normalised). lse_parts: device float32 [num_parts, num_rows], natural
 *   log, -inf for an empty part. o: device [num_rows, head_dim] T, 16-byte
 *   aligned. lse: device float32 [num_rows] or NULL. All parts empty gives
 *   o = 0, lse = -inf.
 */
pd_status pd_merge_states(const float* o_parts, const float* lse_parts, int num_parts,
                          int num_rows, int head_dim, void* o, float* lse, pd_dtype dtype,
                          void* stream);

/* Zero the status header of a workspace (enqueued on stream). */
pd_status pd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read the sticky status word of a workspace into *flags (host). Synchronizes
 * `stream`. The word is not cleared; pd_workspace_init() clears it.
 */
pd_status pd_read_device_flags(const void* workspace, int32_t* flags, void* stream);

/*
 * Plain copy kernel (16-byte vector loads and stores, grid sized to the SM
 * count), used to measure the achievable HBM bandwidth in the same process as
 * the decode, and to bring a step's small inputs in from pinned host memory.
 * dst and src: device memory or pinned host memory (cudaHostAlloc /
 * cudaMallocHost, which kernels reach at its host address under unified
 * addressing), 16-byte aligned, not overlapping; bytes a multiple of 16.
 * Enqueued on stream; the caller keeps both buffers alive until it is done.
 */
pd_status pd_copy_bytes(void* dst, const void* src, size_t bytes, void* stream);

/*
 * Kernel timing for measurement. While enabled, every call records CUDA
 * events on its stream around each kernel it launches (decode, merge,
 * append). pd_profile_read() synchronizes on those events, returns the
 * summed milliseconds and launch counts per kind since the last read (host
 * pointers; any may be NULL), and starts a new count. Enabling costs two
 * event records per kernel; it is off by default.
 */
pd_status pd_profile_enable(int enable);

/*
 * Test-only failure injection for the bounded waits. While extra_bytes is
 * nonzero (a multiple of 16, at most 1 MiB), every decode call's first warp
 * waits, for its first pipeline stage, for extra_bytes more than its copies
 * deliver. Its wait gives up after its limit (2 s), sets
 * PD_FLAG_WAIT_TIMEOUT in the status word, lets its other stages' copies
 * land, and returns; the outputs of the requests it held are then undefined,
 * and the GPU context stays usable. 0 (the default) turns it off.
 * Process-wide; not for use alongside other decode calls.
 */
pd_status pd_test_inject_wait_timeout(int extra_bytes);
pd_status pd_profile_read(double* decode_ms, int* decode_launches, double* merge_ms,
                          int* merge_launches, double* append_ms, int* append_launches);

/*
 * pd_paged_decode for callers that cannot allocate device memory at call
 * time (no counterpart on the pages: it is a deployment variant of the call
 * above). Typical callers: a plugin inside a host engine that owns all
 * device memory and passes its ops no scratch, or a serving loop that may
 * not call cudaMalloc on its hot path. Arguments are those of
 * pd_paged_decode without the workspace.
 *
 * The split-KV scratch lives in a 16 MiB static device array inside this
 * library, which every device that loads the library holds until the
 * process exits. A shape whose scratch (pd_paged_decode_workspace_bytes)
 * exceeds 16 MiB is rejected with PD_ERR_WORKSPACE before anything is
 * enqueued; the bundled workload shapes need at most ~13 MiB on a 148-SM
 * GB300. This call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Each call that passes its argument checks
 * clears the array's status word and then runs the decode; a call rejected
 * by a check enqueues nothing. The kernels' device-side table checks set
 * PD_FLAG_* bits in that word, which pd_paged_decode_noalloc_flags reads.
 * All calls share one array, so calls whose kernels overlap on the GPU
 * (different streams, or different host threads) race on it: order them on
 * one stream.
 */
pd_status pd_paged_decode_noalloc(const void* q, const void* k_data, const void* v_data,
                                  const int32_t* indices, const int32_t* indptr,
                                  const int32_t* last_page_len, void* o, float* lse, int batch,
                                  int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                                  int num_total_pages, int num_indices, float sm_scale,
                                  pd_dtype dtype, void* stream);

/*
 * The status word of pd_paged_decode_noalloc's built-in scratch on the
 * current device, read into *flags (host): the PD_FLAG_* bits that the last
 * pd_paged_decode_noalloc call enqueued before this one set (a bad page id,
 * last_page_len or indptr; a wait that ran out, after which the outputs are
 * invalid). Synchronizes `stream`: enqueue it after that call, on the same
 * stream. Allocates nothing. The word is cleared by the next noalloc call.
 */
pd_status pd_paged_decode_noalloc_flags(int32_t* flags, void* stream);

/* Message for the last error status returned on this host thread ("" if none). */
const char* pd_last_error_string(void);

/* PD_VERSION of the built library. */
int pd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDECODE_H */
