// The walk over one warp's range of positions, shared by the decode kernels.
//
// A position is one (kv head, head tile, listed page) triple: the pages of the
// table are visited once per (kv head, head tile) "pass", in table order, and
// position p is page p % n_pos of pass p / n_pos. A warp owns the positions
// [p0, pend). Request b owns, in every pass, the positions
// [indptr[b], indptr[b+1]) of the table (batch_paged_decode.rs, "Layout":
// indptr is a prefix sum into indices; the last page holds last_page_len
// rows). The contiguous cache is walked the same way with each request's rows
// cut into virtual pages of `vpage` rows.
//
// The walk describes 32 positions at a time, one per lane, so that the
// per-position work (finding the request, reading the page id, the
// last-page length, the flags) runs in parallel; emitting a chunk then costs a
// few shuffles. Page ids of the next window are loaded one window ahead.
#pragma once

#include "pd_device.cuh"

namespace pd {

constexpr int kTableMax = 512;  // requests whose indptr / last_page_len are staged in smem

// Chunk metadata flags. kAppendRow marks the chunk whose last row is the
// request's new row in a fused append + decode.
constexpr int kSegStart = 1, kSegEnd = 2, kSegComplete = 4, kEndOfWork = 8, kAppendRow = 16;
constexpr int kKhShift = 5;  // e_khf = kv head << kKhShift | flags

__host__ __device__ constexpr int round_up(int x, int m) { return (x + m - 1) / m * m; }

inline constexpr int table_bytes_for(bool staged) {
    return staged ? round_up((2 * kTableMax + 1) * 4, 1024) : 0;
}

// One chunk of up to `chunk_rows` rows of one position.
struct Chunk {
    int slab;   // outer index of the K/V slab: page id (paged) or request (contiguous)
    int kh;     // kv head
    int row0;   // first row of the chunk within the (slab, kv head) rows
    int rows;   // valid rows in the chunk (0 .. chunk_rows)
    int flags;  // kSegStart / kSegEnd / kSegComplete
    int qrow;   // first q / o row of the group: b * num_qo_heads + first head of the tile
    int seg;    // segment id: pass * batch + b
};

// Variant bits of the decode kernels (compile-time, one instantiation each).
constexpr int kVarFused = 1;  // the fused append (DecodeArgs::k_new set)
constexpr int kVarNhd = 2;    // contiguous cache in NHD order [batch, max_kv_len, Hk, D]
constexpr int kVarFp8 = 4;    // E4M3 K/V pools with per-kv-head scales (CUDA-core kernel, paged)

// Index, in head_dim-element rows, of row `row` of kv head kh in slab `slab`:
// HND [slab, kv head, row] (pages and the HND contiguous cache) or NHD
// [slab, row, kv head] (the token-major contiguous cache).
template <bool kNhd>
__device__ __forceinline__ size_t kv_row(const DecodeArgs& a, int slab, int kh, long long row) {
    if constexpr (kNhd)
        return (size_t(slab) * size_t(a.slab_rows) + size_t(row)) * size_t(a.num_kv_heads) + size_t(kh);
    else
        return (size_t(slab) * size_t(a.num_kv_heads) + size_t(kh)) * size_t(a.slab_rows) + size_t(row);
}

// The unit that holds position p: share p / ppw, split into a head and
// `pieces` tail pieces of tail / pieces positions (the last one takes the
// remainder) when tail > 0 (see DecodeArgs::tail).
__device__ __forceinline__ long long unit_of(long long p, long long ppw, int tail, int pieces) {
    const long long sh = p / ppw;
    if (tail == 0) return sh;
    const long long r = p - sh * ppw, head = ppw - tail;
    if (r < head) return (1 + pieces) * sh;
    const long long j = min((r - head) / (tail / pieces), (long long)pieces - 1);
    return (1 + pieces) * sh + 1 + j;
}

// kFused: the decode carries the fused append (DecodeArgs::k_new is set);
// only then are new-row chunks marked.
template <bool kFused>
struct Walk {
    const DecodeArgs& a;
    const int* s_indptr;
    const int* s_lpl;
    long long p0, pend;
    int lane;
    bool contiguous, staged;

    // current window: lane k describes position wbase + k
    long long wbase;
    unsigned mask;  // lanes whose position belongs to a request
    int cur, j;     // lane being emitted, chunk within its position
    int nxt;        // prefetched page id of position wbase + 32 + lane
    int e_slab, e_row, e_khf, e_valid, e_qrow, e_seg;  // e_khf = kh << kKhShift | flags

    __device__ __forceinline__ Walk(const DecodeArgs& args, const int* si, const int* sl, long long p0_,
                                    long long pend_, int lane_)
        : a(args), s_indptr(si), s_lpl(sl), p0(p0_), pend(pend_), lane(lane_), contiguous(args.contiguous != 0),
          staged(args.table_bytes > 0), wbase(p0_), mask(0), cur(0), j(0), nxt(-1),
          e_slab(0), e_row(0), e_khf(0), e_valid(0), e_qrow(0), e_seg(0) {}

    // Walk a new range whose first two windows of page ids were loaded ahead
    // (see TailClaim).
    __device__ __forceinline__ void restart_loaded(long long p0_, long long pend_, int pg, int pg_next) {
        p0 = p0_;
        pend = pend_;
        wbase = p0_;
        cur = 0;
        j = 0;
        nxt = pg_next;
        build(p0_, pg);
    }

    // Positions of the current range not emitted yet (an upper bound: some
    // may belong to no request).
    __device__ __forceinline__ long long left() const { return pend - (wbase + cur); }

    // Page id of position p (paged store), -1 outside the range.
    __device__ __forceinline__ int load_page(long long p) const {
        if (contiguous || p >= pend) return -1;
        return __ldg(a.indices + int(p % a.n_pos));
    }

    __device__ __forceinline__ int indptr_at(int b) const { return staged ? s_indptr[b] : __ldg(a.indptr + b); }

    __device__ __forceinline__ void range_of(int b, int* lo, int* hi) const {
        if (contiguous)
            request_range(b, a.n_pos, true, a.npv, 0, 0, lo, hi);
        else
            request_range(b, a.n_pos, false, 0, indptr_at(b), indptr_at(b + 1), lo, hi);
    }

    // Valid rows of request b's last page, clamped to [0, page_size] (flagged if outside).
    __device__ __forceinline__ int last_len(int b) const {
        if (contiguous) return a.valid_kv_len - (a.npv - 1) * a.vpage;
        int v = staged ? s_lpl[b] : __ldg(a.last_page_len + b);
        if (v < 0 || v > a.page_size) {
            atomicOr(a.flags, kFlagBadLastPageLen);
            v = v < 0 ? 0 : a.page_size;
        }
        return v;
    }

    // First request whose range ends after position i (batch if none).
    __device__ __forceinline__ int find_request(int i) const {
        if (contiguous) return min(i / a.npv, a.batch);
        int lo = 0, hi = a.batch;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (indptr_at(mid + 1) > i) hi = mid;
            else lo = mid + 1;
        }
        return lo;
    }

    // Describe positions base .. base + 31, one per lane; pg is this lane's page id.
    __device__ __forceinline__ void build(long long base, int pg) {
        const long long p = base + lane;
        bool has = false;
        e_slab = 0, e_row = 0, e_khf = 0, e_valid = 0, e_qrow = 0, e_seg = 0;
        if (p < pend) {
            const int N = a.n_pos;
            const int sh = int(p / N), i = int(p % N);
            const int b = find_request(i);
            int lo = 0, hi = 0;
            if (b < a.batch) range_of(b, &lo, &hi);
            if (b < a.batch && i >= lo && i < hi) {
                has = true;
                const int kh = sh / a.head_tiles, ht = sh % a.head_tiles;
                const bool last = i == hi - 1;
                int fl = 0;
                if (contiguous) {
                    e_valid = last ? last_len(b) : a.vpage;
                    e_slab = b;
                    e_row = (i - lo) * a.vpage;
                    if (kFused && last && e_valid > 0) fl |= kAppendRow;
                } else {
                    e_valid = last ? last_len(b) : a.page_size;
                    if (pg < 0 || pg >= a.num_total_pages) {
                        atomicOr(a.flags, kFlagBadPage);
                        e_valid = 0;
                        pg = 0;
                    }
                    e_slab = pg;
                    if (kFused && last) {
                        // The new row goes to row last_page_len - 1; a length
                        // outside [1, page_size] or a bad page id skips it.
                        const int raw = staged ? s_lpl[b] : __ldg(a.last_page_len + b);
                        if (raw == 0) atomicOr(a.flags, kFlagBadLastPageLen);
                        if (e_valid > 0 && raw >= 1 && raw <= a.page_size) fl |= kAppendRow;
                    }
                }
                if (i == lo || p == p0) fl |= kSegStart;
                if (i == hi - 1 || p == pend - 1) fl |= kSegEnd;
                if ((long long)sh * N + lo >= p0 && (long long)sh * N + hi <= pend) fl |= kSegComplete;
                e_khf = (kh << kKhShift) | fl;
                e_qrow = b * a.num_qo_heads + kh * a.group + ht * a.heads_per_tile;
                e_seg = sh * a.batch + b;
            }
        }
        mask = __ballot_sync(kFull, has);
    }

    // Issue the page-id loads of the first two windows (before any other set-up).
    __device__ __forceinline__ int prefetch_first() {
        nxt = load_page(p0 + 32 + lane);
        return load_page(p0 + lane);
    }

    // Start pulling the K/V slabs of this warp's first `count` positions into
    // L2 as soon as their page ids are known, before the page table needed to
    // describe them has been staged. Whole slabs: pages hold page_size rows;
    // contiguous slabs are clipped to the cache.
    // In NHD order the rows of one kv head are Hk rows apart: the span from
    // the first to the last is prefetched (other heads' rows included).
    template <bool kNhd>
    __device__ __forceinline__ void prefetch_first_slabs(int pg, int count, size_t row_bytes) {
        const long long p = p0 + lane;
        if (lane >= count || p >= pend) return;
        const int sh = int(p / a.n_pos), i = int(p % a.n_pos);
        const int kh = sh / a.head_tiles;
        size_t row;
        long long rows;
        if (contiguous) {
            const int b = i / a.npv;
            if (b >= a.batch) return;  // a padding position (unit_transpose)
            const long long r0 = (long long)(i % a.npv) * a.vpage;
            rows = min((long long)a.vpage, a.slab_rows - r0);
            row = kv_row<kNhd>(a, b, kh, r0);
        } else {
            if (pg < 0 || pg >= a.num_total_pages) return;
            rows = a.page_size;
            row = kv_row<false>(a, pg, kh, 0);
        }
        if (rows <= 0) return;
        if constexpr (kNhd) rows = (rows - 1) * a.num_kv_heads + 1;
        const uint32_t bytes = uint32_t(rows * (long long)row_bytes);
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.k) + row * row_bytes, bytes);
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.v) + row * row_bytes, bytes);
    }

    // Copy indptr and last_page_len into shared memory. The loads are issued
    // first and stored after `overlap()` runs, so that their latency hides it.
    template <class F>
    __device__ __forceinline__ void stage_table(int* si, int* sl, F overlap) {
        constexpr int kPer = (kTableMax + 1 + 255) / 256;  // entries per thread at 256 threads
        int vi[kPer], vl[kPer];
        const int nt = blockDim.x;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int x = threadIdx.x + k * nt;
            vi[k] = (staged && x <= a.batch) ? __ldg(a.indptr + x) : 0;
            vl[k] = (staged && x < a.batch) ? __ldg(a.last_page_len + x) : 0;
        }
        overlap();
        if (!staged) return;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int x = threadIdx.x + k * nt;
            if (x <= a.batch) si[x] = vi[k];
            if (x < a.batch) sl[x] = vl[k];
        }
        // entries past kPer * blockDim (only with fewer than 256 threads)
        for (int x = threadIdx.x + kPer * nt; x <= a.batch; x += nt) {
            si[x] = __ldg(a.indptr + x);
            if (x < a.batch) sl[x] = __ldg(a.last_page_len + x);
        }
    }

    // The next chunk of at most CR rows; false when the range is exhausted.
    // Move `cur` to the next lane whose position belongs to a request,
    // describing further windows as needed; false when the range is exhausted.
    __device__ __forceinline__ bool seek() {
        while (wbase < pend) {
            const unsigned rest = cur < 32 ? (mask >> cur) : 0u;
            if (rest != 0u) {
                cur += __ffs(rest) - 1;
                return true;
            }
            wbase += 32;
            cur = 0;
            j = 0;
            if (wbase >= pend) break;
            const int pg = nxt;
            nxt = load_page(wbase + 32 + lane);
            build(wbase, pg);
        }
        return false;
    }

    template <int CR>
    __device__ __forceinline__ bool next(Chunk* ck) {
        if (!seek()) return false;
        const int valid = __shfl_sync(kFull, e_valid, cur);
        const int khf = __shfl_sync(kFull, e_khf, cur);
        ck->slab = __shfl_sync(kFull, e_slab, cur);
        ck->row0 = __shfl_sync(kFull, e_row, cur) + j * CR;
        ck->qrow = __shfl_sync(kFull, e_qrow, cur);
        ck->seg = __shfl_sync(kFull, e_seg, cur);
        ck->kh = khf >> kKhShift;
        const int nck = valid > CR ? (valid + CR - 1) / CR : 1;
        int rows = valid - j * CR;
        ck->rows = rows < 0 ? 0 : (rows > CR ? CR : rows);
        int flags = khf & kSegComplete;
        if (j == 0) flags |= khf & kSegStart;
        if (j == nck - 1) flags |= khf & (kSegEnd | kAppendRow);
        ck->flags = flags;
        if (++j == nck) {
            j = 0;
            ++cur;
        }
        return true;
    }
};

// Dynamic tails (DecodeArgs::tail). A warp claims the next tail piece not
// yet taken while its current range still has a few positions to go, and
// requests that piece's first page ids at once: when the range runs out, the
// piece's first chunk follows without waiting for the claim or the ids.
// (Claiming only when the range had run out left each warp ~4 us without
// data per tail on the Llama-shaped batch: the counter's round trip, the page
// ids' round trip, then the first copy's.)
struct TailClaim {
    bool held = false;  // a piece is claimed and its ids requested
    long long t0 = 0, t1 = 0, unit = 0;
    int pg = -1, pg_next = -1;  // page ids of positions t0 + lane and t0 + 32 + lane

    // Claim the next piece not yet taken; false when none is left. Called by
    // the whole warp.
    __device__ __forceinline__ bool claim(const DecodeArgs& a, int lane) {
        const long long ppw = a.pos_per_warp;
        const int kp = a.tail_pieces;
        const long long n_pieces = (a.total_pos + ppw - 1) / ppw * kp;
        const long long piece = a.tail / kp;
        for (;;) {
            unsigned t = 0;
            if (lane == 0) t = atomicAdd(a.tail_ctl, 1u);
            t = __shfl_sync(kFull, t, 0);
            if ((long long)t >= n_pieces) return held = false;
            const long long sh = (long long)t / kp, jp = (long long)t % kp;
            t0 = sh * ppw + (ppw - a.tail) + jp * piece;
            t1 = min(jp == kp - 1 ? (sh + 1) * ppw : t0 + piece, a.total_pos);
            if (t0 >= t1) continue;  // past the last position
            unit = (1 + kp) * sh + 1 + jp;
            const bool paged = a.contiguous == 0;
            pg = (paged && t0 + lane < t1) ? __ldg(a.indices + int((t0 + lane) % a.n_pos)) : -1;
            pg_next = (paged && t0 + 32 + lane < t1) ? __ldg(a.indices + int((t0 + 32 + lane) % a.n_pos)) : -1;
            return held = true;
        }
    }
};

// The producer's next chunk, with the tails: when `walk` runs out, it moves on
// to the claimed tail piece (setting *unit), claiming a new one while the
// current range has at most `ahead` positions left. *tails_left turns false
// once no piece is left to claim. Called by the whole warp.
template <int CR, class W>
__device__ __forceinline__ bool next_with_tails(const DecodeArgs& a, W& walk, TailClaim& tc, bool* tails_left,
                                                long long* unit, int ahead, int lane, Chunk* ck) {
    bool have = walk.template next<CR>(ck);
    while (!have && *tails_left) {
        if (!tc.held && !tc.claim(a, lane)) {
            *tails_left = false;
            break;
        }
        walk.restart_loaded(tc.t0, tc.t1, tc.pg, tc.pg_next);
        *unit = tc.unit;
        tc.held = false;
        have = walk.template next<CR>(ck);
    }
    if (have && *tails_left && !tc.held && walk.left() <= ahead && !tc.claim(a, lane)) *tails_left = false;
    return have;
}

// Every warp of a grid with tails calls this once, after its last chunk; the
// last one resets the tail counters for the next call (no warp takes a piece
// after it has counted itself finished).
__device__ __forceinline__ void tails_finished(const DecodeArgs& a, int nwarps, int lane) {
    if (a.tail == 0 || lane != 0) return;
    __threadfence();
    const unsigned warps = gridDim.x * unsigned(nwarps);
    if (atomicAdd(a.tail_ctl + 1, 1u) == warps - 1u) {
        __threadfence();
        atomicExch(a.tail_ctl, 0u);
        atomicExch(a.tail_ctl + 1, 0u);
    }
}

// Fused append: the whole warp writes request b's new K and V rows for kv
// head ck.kh into the chunk's last row (row ck.row0 + ck.rows - 1 of its
// slab), then fences them so that the chunk's copy, issued afterwards by
// lane 0, reads them. Every warp whose chunk holds the row writes it (the same
// bytes), so no warp depends on another's store.
template <bool kNhd>
__device__ __forceinline__ void write_new_row(const DecodeArgs& a, const Chunk& ck, int lane, size_t row_bytes) {
    const int b = ck.seg % a.batch;
    const size_t src = (size_t(b) * a.num_kv_heads + ck.kh) * row_bytes;
    const size_t dst = kv_row<kNhd>(a, ck.slab, ck.kh, ck.row0 + ck.rows - 1) * row_bytes;
    uint8_t* kd = static_cast<uint8_t*>(const_cast<void*>(a.k)) + dst;
    uint8_t* vd = static_cast<uint8_t*>(const_cast<void*>(a.v)) + dst;
    const uint8_t* ks = static_cast<const uint8_t*>(a.k_new) + src;
    const uint8_t* vs = static_cast<const uint8_t*>(a.v_new) + src;
    for (size_t off = size_t(lane) * 16; off < row_bytes; off += 32 * 16) {
        *reinterpret_cast<uint4*>(kd + off) = __ldg(reinterpret_cast<const uint4*>(ks + off));
        *reinterpret_cast<uint4*>(vd + off) = __ldg(reinterpret_cast<const uint4*>(vs + off));
    }
    fence_proxy_async_global();
    __syncwarp();
}

}  // namespace pd
