// CPU oracle for batched decode attention over a paged KV cache.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
// load this file; only tests/, the smoke check and the benchmark's CPU
// baseline use it. It shares no code, header, table or helper with the CUDA
// library: it decodes the input bytes itself and computes each result from
// its plain definition, slowly, in double precision.
//
// Sources (each function cites the passage it follows):
//  [P3] baracuda-kernels 0.0.1-alpha.68, src/attention/batch_paged_decode.rs:
//       module doc "Layout" (HND pages, indices/indptr/last_page_len, q/o/lse
//       shapes, lse always f32) and "Constraints" (GQA group must be an
//       integer); PagedKvCacheDescriptor / BatchPagedDecodeDescriptor fields.
//  [P1] ferrum-kernels 0.7.7, src/backend/cuda/decode_attention.rs: module doc
//       (scores, stable softmax, scores times V) and the decode_attention
//       arguments (contiguous k_cache [num_kv_heads, max_kv_len, head_dim],
//       valid_kv_len, scale).
//  [P2] ferrox-cuda 0.15.2, src/attn.rs: gqa_decode (the q-head to kv-head
//       map kv_h = h / (n_heads / n_kv_heads); zero output for an empty cache).
//
// ORACLE_MUTANT (compile-time, never set in a normal build) plants one known
// mistake; tests/test_oracle_mutants.py builds each mutant and checks that the
// pins in tests/test_oracle.py fail on it.
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
//
// Readings where the pages are silent (each also listed in the design notes):
//  - lse is the natural log of the sum of exp(scaled score): lse = m + ln(Z).
//  - sm_scale multiplies q.k before the softmax, so lse is over scaled scores.
//  - token t of a request is row t % page_size of its (t / page_size)-th listed
//    page; every listed page but the last is full.
//  - a request with no valid rows returns o = 0 and lse = -inf.
//  - the caller's f32 sm_scale is used as given, widened to double.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
double from_f16_bits(uint16_t h) {
    const int sign = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = std::ldexp(double(f), -24);  // subnormal: f * 2^-24
    else if (e == 31)
        v = f ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
    else
        v = std::ldexp(double(f | 0x400), e - 25);  // (1024 + f) * 2^(e - 15 - 10)
    return sign ? -v : v;
}

// bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.
double from_bf16_bits(uint16_t b) {
    const int sign = b >> 15, e = (b >> 7) & 0xff, f = b & 0x7f;
    double v;
    if (e == 0)
        v = std::ldexp(double(f), -133);  // subnormal: f * 2^(-126 - 7)
    else if (e == 255)
        v = f ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
    else
        v = std::ldexp(double(f | 0x80), e - 134);  // (128 + f) * 2^(e - 127 - 7)
    return sign ? -v : v;
}

double from_f32_bits(uint32_t u) {
    float f;
    std::memcpy(&f, &u, 4);
    return double(f);
}

struct View {
    const void* p;
    int dtype;
    double at(size_t i) const {
        if (dtype == DT_F32) {
            uint32_t u;
            std::memcpy(&u, static_cast<const uint8_t*>(p) + 4 * i, 4);
            return from_f32_bits(u);
        }
        uint16_t h;
        std::memcpy(&h, static_cast<const uint8_t*>(p) + 2 * i, 2);
        return dtype == DT_F16 ? from_f16_bits(h) : from_bf16_bits(h);
    }
};

size_t elem_bytes(int dtype) { return dtype == DT_F32 ? 4 : 2; }

// FP8 E4M3 as the OCP 8-bit floating point specification (OFP8) defines it:
// sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
// the subnormals (m / 8) * 2^-6; S.1111.111 is NaN; there is no infinity, so
// S.1111.110 = 448 is the largest finite magnitude.
double e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
    const int bias = ORACLE_MUTANT == 12 ? 8 : 7;
    const double v = e == 0 && ORACLE_MUTANT != 14 ? std::ldexp(m / 8.0, 1 - bias) : std::ldexp(1.0 + m / 8.0, e - bias);
    return s ? -v : v;
}

// Round to E4M3, nearest with ties to the even code, finite values past 448
// (and infinities) saturating to +-448, NaN to the NaN code 0x7F. By brute
// force over the 127 non-negative finite codes (their values increase with
// the code, and of two neighbours exactly one has an even code).
uint8_t e4m3_round(float x) {
    if (std::isnan(x)) return 0x7F;
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    const double a = std::fabs(double(x));
    if (std::isinf(a)) return sign | 0x7E;
    if (ORACLE_MUTANT == 16 && a > 464.0) return sign | 0x7F;  // mutant 16: overflow to NaN
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 0x7E; ++c) {
        const double err = std::fabs(e4m3_value(uint8_t(c)) - a);
        if (err < best_err || (err == best_err && (ORACLE_MUTANT == 15 || (c & 1) == 0))) best = c, best_err = err;
    }
    return uint8_t(sign | best);
}

template <class F>
void parallel_for(long n, int nthreads, F f) {
    if (nthreads <= 0) nthreads = int(std::thread::hardware_concurrency());
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = int(n > 0 ? n : 1);
    if (nthreads == 1) {
        for (long i = 0; i < n; ++i) f(i);
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t)
        pool.emplace_back([=] {
            for (long i = t; i < n; i += nthreads) f(i);
        });
    for (auto& th : pool) th.join();
}

// Attention of one query row over n keys given by the accessors, two passes:
// pass 1 takes m = max_t s_t, pass 2 sums w_t = exp(s_t - m) and w_t * v_t.
// [P1] module doc steps 1-3; [P3] "Layout" (o row and f32 lse per row).
template <class KAt, class VAt>
void attend(const View& q, size_t q_off, long n, int D, double scale, KAt k_at, VAt v_at,
            double* o, double* lse) {
    if (n <= 0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *lse = ORACLE_MUTANT == 18 ? 0.0 : -std::numeric_limits<double>::infinity();
        return;
    }
    std::vector<double> s(static_cast<size_t>(n));
    for (long t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q.at(q_off + d) * k_at(t, d);
        s[size_t(t)] = (ORACLE_MUTANT == 1 ? 1.0 : scale) * dot;  // mutant 1: scale dropped
    }
    double m = s[0];
    for (long t = 1; t < n; ++t) m = s[size_t(t)] > m ? s[size_t(t)] : m;
    double Z = 0.0;
    std::vector<double> acc(size_t(D), 0.0);
    for (long t = 0; t < n; ++t) {
        const double w = std::exp(s[size_t(t)] - m);
        Z += w;
        for (int d = 0; d < D; ++d) acc[size_t(d)] += w * (ORACLE_MUTANT == 2 ? k_at(t, d) : v_at(t, d));
    }
    for (int d = 0; d < D; ++d) o[d] = ORACLE_MUTANT == 3 ? acc[size_t(d)] : acc[size_t(d)] / Z;
    *lse = ORACLE_MUTANT == 4 ? m + std::log2(Z) : m + std::log(Z);
}

}  // namespace

// Shared by the paged decodes: validates the table ([P3] "Layout") and runs
// attend() for every (request, q head), with kval(i, kh) / vval(i, kh) the
// value of element i of the K / V pool, which belongs to kv head kh.
template <class KV, class VV>
int paged_decode_values(const void* q, int q_dtype, KV kval, VV vval, const int32_t* indices,
                        const int32_t* indptr, const int32_t* last_page_len, int batch, int num_qo_heads,
                        int num_kv_heads, int head_dim, int page_size, int num_total_pages, long num_indices,
                        float sm_scale, double* o_out, double* lse_out, int nthreads) {
    if (batch <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
        num_total_pages <= 0 || q_dtype < 0 || q_dtype > 2)
        return 1;
    if (num_qo_heads % num_kv_heads != 0) return 1;  // [P3] "Constraints": integer group
    if (indptr[0] < 0) return 2;
    for (int b = 0; b < batch; ++b) {
        if (indptr[b + 1] < indptr[b]) return 2;
        if (indptr[b + 1] > indptr[b] && (last_page_len[b] < 0 || last_page_len[b] > page_size)) return 2;
    }
    if (indptr[batch] > num_indices) return 2;
    for (long i = indptr[0]; i < indptr[batch]; ++i)
        if (indices[i] < 0 || indices[i] >= num_total_pages) return 2;

    const int group = num_qo_heads / num_kv_heads;
    const View Q{q, q_dtype};
    const double scale = double(sm_scale);
    parallel_for(long(batch) * num_qo_heads, nthreads, [&](long bh) {
        const int b = int(bh / num_qo_heads), h = int(bh % num_qo_heads);
        const int kh = ORACLE_MUTANT == 5 ? h % num_kv_heads : h / group;  // [P2] gqa_decode: kv_h = h / group_size
        const long np = indptr[b + 1] - indptr[b];
        const long n = np == 0 ? 0 : (np - 1) * page_size + (ORACLE_MUTANT == 6 ? page_size : last_page_len[b]);
        auto addr = [&](long t, int d) {
            const size_t page = size_t(indices[indptr[b] + t / page_size]);
            const size_t row = size_t(ORACLE_MUTANT == 7 ? page_size - 1 - t % page_size : t % page_size);
            return ((page * num_kv_heads + kh) * page_size + row) * head_dim + size_t(d);
        };
        attend(Q, size_t(bh) * head_dim, n, head_dim, scale,
               [&](long t, int d) { return kval(addr(t, d), kh); },
               [&](long t, int d) { return vval(addr(t, d), kh); },
               o_out + size_t(bh) * head_dim, lse_out + bh);
    });
    return 0;
}

extern "C" {

// Decode nelem elements of a raw array of dtype into doubles.
int oracle_decode_elements(const void* src, int dtype, long nelem, double* out) {
    if (dtype < 0 || dtype > 2 || nelem < 0) return 1;
    View v{src, dtype};
    for (long i = 0; i < nelem; ++i) out[i] = v.at(size_t(i));
    return 0;
}

// Batched decode over the paged store, [P3] "Layout":
//   k_data/v_data [num_total_pages, num_kv_heads, page_size, head_dim] (HND),
//   request b owns pages indices[indptr[b] .. indptr[b+1]), its last page holds
//   last_page_len[b] valid rows, so kv_len = (np - 1) * page_size + last_page_len.
// q [batch, num_qo_heads, head_dim]; o_out [batch, num_qo_heads, head_dim] and
// lse_out [batch, num_qo_heads] are written in double.
// Returns 0, or 1 for a bad descriptor / 2 for a bad page table.
int oracle_paged_decode(const void* q, const void* k_data, const void* v_data,
                        const int32_t* indices, const int32_t* indptr, const int32_t* last_page_len,
                        int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                        int num_total_pages, long num_indices, float sm_scale, int dtype,
                        double* o_out, double* lse_out, int nthreads) {
    if (dtype < 0 || dtype > 2) return 1;
    const View K{k_data, dtype}, V{v_data, dtype};
    return paged_decode_values(
        q, dtype, [&](size_t i, int) { return K.at(i); }, [&](size_t i, int) { return V.at(i); }, indices, indptr,
        last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices,
        sm_scale, o_out, lse_out, nthreads);
}

// The paged decode over an FP8 pool: K and V pages hold E4M3 codes (one byte
// per element, same HND layout), and element value = e4m3_value(code) *
// k_scale[kh] (v_scale[kh] for V), kh the element's kv head. q and o are
// q_dtype (f16 or bf16). This is this library's own extension, not a layout
// of the pages: a per-kv-head scale is the plainest scheme that keeps the
// pool one byte per element.
int oracle_paged_decode_fp8(const void* q, const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scale,
                            const float* v_scale, const int32_t* indices, const int32_t* indptr,
                            const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads,
                            int head_dim, int page_size, int num_total_pages, long num_indices, float sm_scale,
                            int q_dtype, double* o_out, double* lse_out, int nthreads) {
    if (q_dtype != DT_F16 && q_dtype != DT_BF16) return 1;
    const float* vs = ORACLE_MUTANT == 13 ? k_scale : v_scale;
    return paged_decode_values(
        q, q_dtype, [&](size_t i, int kh) { return e4m3_value(k_codes[i]) * double(k_scale[kh]); },
        [&](size_t i, int kh) { return e4m3_value(v_codes[i]) * double(vs[kh]); }, indices, indptr,
        last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, num_indices,
        sm_scale, o_out, lse_out, nthreads);
}

// E4M3 codes of values / per-element conversions, for the pins.
int oracle_e4m3_values(const uint8_t* codes, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
    return 0;
}
int oracle_e4m3_round(const float* x, long n, uint8_t* out) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_round(x[i]);
    return 0;
}

// Row index (in head_dim-element rows) of token t, kv head kh, request b in a
// contiguous cache of one of two layouts:
//   layout 0, HND: [batch, num_kv_heads, max_kv_len, head_dim] ([P1] decode_attention
//                  k_cache [num_kv_heads, max_kv_len, head_dim], batch in front);
//   layout 1, NHD: [batch, max_kv_len, num_kv_heads, head_dim] ([P2] gqa_decode:
//                  token t of kv head kv_h starts at (t * n_kv_heads + kv_h) * head_dim,
//                  batch in front).
static size_t contiguous_row(int layout, int b, int kh, long t, int num_kv_heads, long max_kv_len) {
    if (layout == 1 && ORACLE_MUTANT != 11)
        return (size_t(b) * size_t(max_kv_len) + size_t(t)) * size_t(num_kv_heads) + size_t(kh);
    return (size_t(b) * size_t(num_kv_heads) + size_t(kh)) * size_t(max_kv_len) + size_t(t);
}

// Decode over a contiguous cache, [P1] decode_attention arguments, with a batch
// dimension in front; rows [0, valid_kv_len) valid for every request; layout as
// in contiguous_row. A separate loop from the paged walk on purpose: the two
// paths agreeing is itself a check.
int oracle_contiguous_decode(const void* q, const void* k_cache, const void* v_cache, int batch,
                             int num_qo_heads, int num_kv_heads, int head_dim, long max_kv_len,
                             long valid_kv_len, float sm_scale, int dtype, int layout, double* o_out,
                             double* lse_out, int nthreads) {
    if (batch <= 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_kv_len <= 0 ||
        valid_kv_len < 0 || valid_kv_len > max_kv_len || dtype < 0 || dtype > 2 || layout < 0 || layout > 1)
        return 1;
    if (num_qo_heads % num_kv_heads != 0) return 1;
    const int group = num_qo_heads / num_kv_heads;
    const View Q{q, dtype}, K{k_cache, dtype}, V{v_cache, dtype};
    const double scale = double(sm_scale);
    parallel_for(long(batch) * num_qo_heads, nthreads, [&](long bh) {
        const int b = int(bh / num_qo_heads), h = int(bh % num_qo_heads);
        const int kh = h / group;
        auto addr = [&](long t, int d) {
            return contiguous_row(layout, b, kh, t, num_kv_heads, max_kv_len) * size_t(head_dim) + size_t(d);
        };
        attend(Q, size_t(bh) * head_dim, ORACLE_MUTANT == 19 ? max_kv_len : valid_kv_len, head_dim, scale,
               [&](long t, int d) { return K.at(addr(t, d)); },
               [&](long t, int d) { return V.at(addr(t, d)); },
               o_out + size_t(bh) * head_dim, lse_out + bh);
    });
    return 0;
}

// Paged append on a host mirror of the pool: for every request b and kv head h
// the row k_new[b, h, :] goes to row last_page_len[b] - 1 of page
// indices[indptr[b+1] - 1], head h; the same for v. The caller has already
// updated the table ([P3] "Companion plans": the append writes the new K/V
// slices into the paged store; the caller owns the table).
// Returns 0, 1 for a bad descriptor, 2 for a bad table entry.
int oracle_paged_append(const void* k_new, const void* v_new, void* k_data, void* v_data,
                        const int32_t* indices, const int32_t* indptr, const int32_t* last_page_len,
                        int batch, int num_kv_heads, int head_dim, int page_size, int num_total_pages,
                        int dtype) {
    if (batch <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_total_pages <= 0 ||
        dtype < 0 || dtype > 2)
        return 1;
    const size_t eb = elem_bytes(dtype), row = size_t(head_dim) * eb;
    for (int b = 0; b < batch; ++b) {
        if (indptr[b + 1] <= indptr[b]) return 2;
        const int slot = ORACLE_MUTANT == 8 ? last_page_len[b] % page_size : last_page_len[b] - 1;
        const int page = indices[indptr[b + 1] - 1];
        if (slot < 0 || slot >= page_size || page < 0 || page >= num_total_pages) return 2;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t dst = ((size_t(page) * num_kv_heads + h) * page_size + size_t(slot)) * row;
            const size_t src = (size_t(b) * num_kv_heads + h) * row;
            std::memcpy(static_cast<uint8_t*>(k_data) + dst, static_cast<const uint8_t*>(k_new) + src, row);
            std::memcpy(static_cast<uint8_t*>(v_data) + dst, static_cast<const uint8_t*>(v_new) + src, row);
        }
    }
    return 0;
}

// Paged append into an FP8 pool: the slot of oracle_paged_append receives
// the codes e4m3_round(x / scale[h]) of the new row, x the exact value of the
// f16 / bf16 element widened to f32 and the division done in f32 (the
// quantisation decision is made in f32 on both sides of a parity test).
// Returns 0, 1 for a bad descriptor, 2 for a bad table entry.
int oracle_paged_append_fp8(const void* k_new, const void* v_new, const float* k_scale, const float* v_scale,
                            uint8_t* k_codes, uint8_t* v_codes, const int32_t* indices, const int32_t* indptr,
                            const int32_t* last_page_len, int batch, int num_kv_heads, int head_dim, int page_size,
                            int num_total_pages, int new_dtype) {
    if (batch <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_total_pages <= 0 ||
        (new_dtype != DT_F16 && new_dtype != DT_BF16))
        return 1;
    const View KN{k_new, new_dtype}, VN{v_new, new_dtype};
    for (int b = 0; b < batch; ++b) {
        if (indptr[b + 1] <= indptr[b]) return 2;
        const int slot = last_page_len[b] - 1;
        const int page = indices[indptr[b + 1] - 1];
        if (slot < 0 || slot >= page_size || page < 0 || page >= num_total_pages) return 2;
        for (int h = 0; h < num_kv_heads; ++h)
            for (int d = 0; d < head_dim; ++d) {
                const size_t dst = ((size_t(page) * num_kv_heads + h) * page_size + size_t(slot)) * head_dim + d;
                const size_t src = (size_t(b) * num_kv_heads + h) * head_dim + d;
                k_codes[dst] = e4m3_round(ORACLE_MUTANT == 17 ? float(KN.at(src)) * k_scale[h]
                                                              : float(KN.at(src)) / k_scale[h]);
                v_codes[dst] = e4m3_round(float(VN.at(src)) / v_scale[h]);
            }
    }
    return 0;
}

// Append to a contiguous cache ([P3] "Companion plans": KvCacheAppendPlan, the
// rank-4 cache with no page table): for every request b and kv head h, token
// `position` of kv head h of request b becomes k_new[b, h, :], the same for v.
// Layout as in contiguous_row. Returns 0 or 1.
int oracle_contiguous_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int batch,
                             int num_kv_heads, int head_dim, long max_kv_len, long position, int dtype,
                             int layout) {
    if (batch <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_kv_len <= 0 || position < 0 ||
        position >= max_kv_len || dtype < 0 || dtype > 2 || layout < 0 || layout > 1)
        return 1;
    const size_t row = size_t(head_dim) * elem_bytes(dtype);
    for (int b = 0; b < batch; ++b)
        for (int h = 0; h < num_kv_heads; ++h) {
            const long pos = ORACLE_MUTANT == 10 ? (position > 0 ? position - 1 : position + 1) : position;
            const size_t dst = contiguous_row(layout, b, h, pos, num_kv_heads, max_kv_len) * row;
            const size_t src = (size_t(b) * num_kv_heads + h) * row;
            std::memcpy(static_cast<uint8_t*>(k_cache) + dst, static_cast<const uint8_t*>(k_new) + src, row);
            std::memcpy(static_cast<uint8_t*>(v_cache) + dst, static_cast<const uint8_t*>(v_new) + src, row);
        }
    return 0;
}

// Merge of attention states computed over disjoint key sets into the state over
// their union: L = ln sum_c exp(lse_c), o = sum_c exp(lse_c - L) * o_c. With
// M = max_c lse_c, L = M + ln sum_c exp(lse_c - M). All parts empty (every
// lse_c = -inf) gives o = 0, lse = -inf.
// o_parts [num_parts, rows, head_dim], lse_parts [num_parts, rows].
int oracle_merge_states(const double* o_parts, const double* lse_parts, int num_parts, long rows,
                        int head_dim, double* o_out, double* lse_out) {
    if (num_parts <= 0 || rows < 0 || head_dim <= 0) return 1;
    const double ninf = -std::numeric_limits<double>::infinity();
    for (long r = 0; r < rows; ++r) {
        double M = ninf;
        for (int c = 0; c < num_parts; ++c) M = lse_parts[size_t(c) * rows + r] > M ? lse_parts[size_t(c) * rows + r] : M;
        double* o = o_out + size_t(r) * head_dim;
        if (M == ninf) {
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            lse_out[r] = ninf;
            continue;
        }
        double S = 0.0;
        for (int c = 0; c < num_parts; ++c) S += std::exp(lse_parts[size_t(c) * rows + r] - M);
        const double L = ORACLE_MUTANT == 20 ? M : M + std::log(S);
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        for (int c = 0; c < num_parts; ++c) {
            const double w = std::exp(ORACLE_MUTANT == 9 ? L - lse_parts[size_t(c) * rows + r] : lse_parts[size_t(c) * rows + r] - L);
            const double* oc = o_parts + (size_t(c) * rows + r) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] += w * oc[d];
        }
        lse_out[r] = L;
    }
    return 0;
}

// Round doubles to the storage type, round-to-nearest-even, for reporting the
// rounding floor of an output. Written from the format definitions.
int oracle_round_to_dtype(const double* x, long n, int dtype, void* out) {
    if (dtype < 0 || dtype > 2) return 1;
    for (long i = 0; i < n; ++i) {
        const double v = x[i];
        if (dtype == DT_F32) {
            const float f = float(v);  // C++ conversion rounds to nearest even
            std::memcpy(static_cast<uint8_t*>(out) + 4 * size_t(i), &f, 4);
            continue;
        }
        const int frac_bits = dtype == DT_F16 ? 10 : 7;
        const int emin = dtype == DT_F16 ? -14 : -126;  // exponent of the smallest normal
        const int emax = dtype == DT_F16 ? 15 : 127;
        const int bias = dtype == DT_F16 ? 15 : 127;
        const uint16_t inf_bits = dtype == DT_F16 ? 0x7c00 : 0x7f80;
        const double maxv = std::ldexp(2.0 - std::ldexp(1.0, -frac_bits), emax);
        const double a = std::fabs(v);
        uint16_t bits;
        if (std::isnan(v)) {
            bits = dtype == DT_F16 ? 0x7e00 : 0x7fc0;
        } else if (a == 0.0) {
            bits = 0;
        } else if (std::isinf(a)) {
            bits = inf_bits;
        } else {
            int e;
            std::frexp(a, &e);  // a = m * 2^e with m in [0.5, 1), so a = 1.f * 2^(e-1)
            int ue = e - 1;
            if (ue < emin) ue = emin;  // subnormals share the quantum of the smallest normal
            const double quantum = std::ldexp(1.0, ue - frac_bits);
            const double r = std::nearbyint(a / quantum) * quantum;  // RNE at that quantum
            if (r > maxv) {
                bits = inf_bits;
            } else if (r < std::ldexp(1.0, emin)) {  // subnormal (or zero) result
                bits = uint16_t(std::ldexp(r, frac_bits - emin));
            } else {
                int re;
                std::frexp(r, &re);
                const int rue = re - 1;
                const uint32_t frac = uint32_t(std::ldexp(r, frac_bits - rue)) - (1u << frac_bits);
                bits = uint16_t((uint32_t(rue + bias) << frac_bits) | frac);
            }
        }
        if (std::signbit(v) && !std::isnan(v)) bits = uint16_t(bits | 0x8000u);
        std::memcpy(static_cast<uint8_t*>(out) + 2 * size_t(i), &bits, 2);
    }
    return 0;
}

int oracle_hardware_threads(void) { return int(std::thread::hardware_concurrency()); }

}  // extern "C"
