"""Seeded synthetic workloads for batched paged-KV decode.

This module makes inputs only: random values (``fill.c``), page tables as a
serving stack's block allocator would build them, and the host-side table
update that precedes a paged append. It computes nothing that the attention
kernels or the oracle compute, and it imports neither of them. Both sides
are fed the same bytes from here.

Layout of what it builds (baracuda-kernels ``batch_paged_decode.rs``, module
doc "Layout"):
  q            [batch, num_qo_heads, head_dim]                element type T
  k_data/v_data [num_total_pages, num_kv_heads, page_size, head_dim]  (HND)
  indices      [num_indices] int32 physical page ids
  indptr       [batch + 1]   int32 prefix sum into ``indices``
  last_page_len[batch]       int32 valid rows of each request's last page

Storage of T on the host: float32 arrays for f32, uint16 bit patterns for
f16 and bf16. Pages that no request uses, and rows at or past
``last_page_len`` in last pages, are filled with NaN so that a kernel that
reads them cannot go unnoticed.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fill.c")
_SO = os.path.join(_HERE, "libwlfill.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
_NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}

# Stream ids: each tensor of a workload draws from its own splitmix64 stream.
STREAMS = {"q": 1, "k": 2, "v": 3, "k_new": 4, "v_new": 5, "k_e4m3": 6, "v_e4m3": 7, "k_scale": 8, "v_scale": 9}


def build(force: bool = False) -> str:
    """Compile fill.c into libwlfill.so next to it (portable C, no ISA flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        lib.wl_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                       ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
        lib.wl_fill_normal.restype = ctypes.c_int
        lib.wl_round_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64]
        lib.wl_round_f32.restype = ctypes.c_int
        lib.wl_fill_e4m3.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_int, ctypes.c_int]
        lib.wl_fill_e4m3.restype = ctypes.c_int
        lib.wl_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wl_splitmix64_at.restype = ctypes.c_uint64
        _lib_handle = lib
    return _lib_handle


def raw_np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def splitmix64_at(key: int, n: int) -> int:
    return int(_lib().wl_splitmix64_at(key, n))


def stream_key(seed: int, stream: str) -> int:
    """Key of one tensor's stream: splitmix64 output number STREAMS[stream] for `seed`."""
    return splitmix64_at(seed, STREAMS[stream])


def normal(shape, dtype: str, key: int, first: int = 0, threads: int | None = None) -> np.ndarray:
    """N(0,1) draws first.. of stream `key`, rounded (RNE) to dtype; raw storage."""
    out = np.empty(shape, dtype=raw_np_dtype(dtype))
    fill_normal(out, dtype, key, first, threads)
    return out


def fill_normal(out: np.ndarray, dtype: str, key: int, first: int = 0, threads: int | None = None):
    assert out.flags.c_contiguous and out.dtype == raw_np_dtype(dtype)
    nthreads = threads or os.cpu_count() or 1
    rc = _lib().wl_fill_normal(out.ctypes.data, DTYPE_CODE[dtype], out.size, key, first, nthreads)
    if rc != 0:
        raise ValueError("wl_fill_normal failed")
    return out


def round_f32(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage type (RNE); identity for f32."""
    values = np.ascontiguousarray(values, dtype=np.float32)
    if dtype == "f32":
        return values.copy()
    out = np.empty(values.shape, dtype=np.uint16)
    if _lib().wl_round_f32(values.ctypes.data, out.ctypes.data, DTYPE_CODE[dtype], values.size) != 0:
        raise ValueError("bad dtype")
    return out


def nan_value(dtype: str):
    if dtype == "e4m3":
        return np.uint8(E4M3_NAN)
    return np.float32(np.nan) if dtype == "f32" else np.uint16(_NAN_BITS[dtype])


# --- FP8 (E4M3) pools -----------------------------------------------------------------------

E4M3_NAN = 0x7F  # S.1111.111 with S = 0


def e4m3_codes(shape, key: int, first: int = 0, e_lo: int = 4, e_hi: int = 9) -> np.ndarray:
    """Random E4M3 codes (uint8): random sign and mantissa, exponent field uniform in
    [e_lo, e_hi] (default: magnitudes 0.125 .. 7.5). Bit fields only, no rounding."""
    out = np.empty(shape, dtype=np.uint8)
    if _lib().wl_fill_e4m3(out.ctypes.data, out.size, key, first, e_lo, e_hi) != 0:
        raise ValueError("wl_fill_e4m3: exponent range must lie in [1, 14]")
    return out


def kv_scales(num_kv_heads: int, key: int, lo: float = 0.05, hi: float = 0.2) -> np.ndarray:
    """Per-kv-head float32 scales lo + (hi - lo) * u, u uniform from stream `key`."""
    u = np.array([(splitmix64_at(key, h) >> 11) / float(1 << 53) for h in range(num_kv_heads)])
    return (lo + (hi - lo) * u).astype(np.float32)


def fp8_pool(w: "Workload"):
    """An E4M3 pool of w's shape and table: codes from their own streams, unused
    rows poisoned with the NaN code, and per-kv-head K and V scales."""
    k = e4m3_codes(w.k_data.shape, stream_key(w.seed, "k_e4m3"))
    v = e4m3_codes(w.v_data.shape, stream_key(w.seed, "v_e4m3"))
    poison_unused(k, v, w.table, "e4m3")
    return (k, v, kv_scales(w.num_kv_heads, stream_key(w.seed, "k_scale")),
            kv_scales(w.num_kv_heads, stream_key(w.seed, "v_scale")))


@dataclass
class PageTable:
    """A request-to-page map built by the caller's block allocator."""

    page_size: int
    num_total_pages: int
    indptr: np.ndarray  # int32 [batch + 1]
    indices: np.ndarray  # int32 [num_indices]
    last_page_len: np.ndarray  # int32 [batch]
    free_pages: list = field(default_factory=list)  # pool pages not in use, in allocation order

    @property
    def batch(self) -> int:
        return len(self.last_page_len)

    @property
    def num_indices(self) -> int:
        return len(self.indices)

    def kv_len(self) -> np.ndarray:
        npg = np.diff(self.indptr).astype(np.int64)
        return np.where(npg > 0, (npg - 1) * self.page_size + self.last_page_len, 0)

    def copy(self) -> "PageTable":
        return PageTable(self.page_size, self.num_total_pages, self.indptr.copy(),
                         self.indices.copy(), self.last_page_len.copy(), list(self.free_pages))


def pages_needed(kv_len, page_size: int) -> np.ndarray:
    kv_len = np.asarray(kv_len, dtype=np.int64)
    return (kv_len + page_size - 1) // page_size


def build_page_table(kv_len, page_size: int, num_total_pages: int, rng: np.random.Generator) -> PageTable:
    """Give each request ceil(kv_len/page_size) pages drawn from a shuffled pool.

    Pages are handed out in the order of one random permutation of the pool,
    so each request's pages are scattered and in no particular physical order.
    """
    kv_len = np.asarray(kv_len, dtype=np.int64)
    npg = pages_needed(kv_len, page_size)
    total = int(npg.sum())
    if total > num_total_pages:
        raise ValueError("pool too small")
    perm = rng.permutation(num_total_pages).astype(np.int32)
    indptr = np.zeros(len(kv_len) + 1, dtype=np.int32)
    indptr[1:] = np.cumsum(npg)
    lpl = np.where(npg > 0, kv_len - (npg - 1) * page_size, 0).astype(np.int32)
    return PageTable(page_size, num_total_pages, indptr, perm[:total].copy(), lpl,
                     [int(p) for p in perm[total:]])


def table_after_append(table: PageTable) -> PageTable:
    """The caller's table update before a one-row paged append to every request.

    A request whose last page is full (or that has no page) takes the next
    free page, which is appended to its page list with one valid row;
    otherwise its last page gains one row. The new row is then the last
    valid row of the last page. (The caller owns the page table and its
    allocator: baracuda-kernels ``batch_paged_decode.rs``, module doc,
    "Companion plans".)
    """
    t = table.copy()
    P = t.page_size
    new_indices = []
    new_indptr = [0]
    lpl = t.last_page_len.copy()
    for b in range(t.batch):
        pages = list(t.indices[t.indptr[b]:t.indptr[b + 1]])
        if len(pages) == 0 or lpl[b] == P:
            if not t.free_pages:
                raise RuntimeError("page pool exhausted")
            pages.append(t.free_pages.pop(0))
            lpl[b] = 1
        else:
            lpl[b] += 1
        new_indices.extend(pages)
        new_indptr.append(len(new_indices))
    t.indices = np.asarray(new_indices, dtype=np.int32)
    t.indptr = np.asarray(new_indptr, dtype=np.int32)
    t.last_page_len = lpl.astype(np.int32)
    return t


def poison_unused(k: np.ndarray, v: np.ndarray, table: PageTable, dtype: str):
    """NaN every pool page no request uses and every row past last_page_len."""
    nanv = nan_value(dtype)
    used = np.zeros(table.num_total_pages, dtype=bool)
    used[table.indices] = True
    k[~used] = nanv
    v[~used] = nanv
    for b in range(table.batch):
        lo, hi = int(table.indptr[b]), int(table.indptr[b + 1])
        if hi > lo:
            last = int(table.indices[hi - 1])
            k[last, :, int(table.last_page_len[b]):, :] = nanv
            v[last, :, int(table.last_page_len[b]):, :] = nanv


@dataclass
class Workload:
    """One synthetic batched paged-decode problem, inputs on the host."""

    name: str
    dtype: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    table: PageTable
    q: np.ndarray
    k_data: np.ndarray
    v_data: np.ndarray
    sm_scale: float
    seed: int
    append_steps: int = 0
    description: str = ""

    @property
    def batch(self) -> int:
        return self.table.batch

    @property
    def page_size(self) -> int:
        return self.table.page_size

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    def kv_bytes(self, table: PageTable | None = None) -> int:
        """K+V bytes a decode must read: valid rows only."""
        t = table or self.table
        return int(t.kv_len().sum()) * self.num_kv_heads * self.head_dim * ELEM_BYTES[self.dtype] * 2

    def qo_bytes(self) -> int:
        return 2 * self.batch * self.num_qo_heads * self.head_dim * ELEM_BYTES[self.dtype]

    def new_rows(self, step: int):
        """k_new, v_new [batch, num_kv_heads, head_dim] appended at append step `step`."""
        n = self.batch * self.num_kv_heads * self.head_dim
        shape = (self.batch, self.num_kv_heads, self.head_dim)
        k = normal(shape, self.dtype, stream_key(self.seed, "k_new"), first=step * n)
        v = normal(shape, self.dtype, stream_key(self.seed, "v_new"), first=step * n)
        return k, v


def make_paged(name, dtype, kv_len, num_qo_heads, num_kv_heads, head_dim, page_size, seed,
               pool_pages=None, pool_slack=0.10, extra_rows=0, append_steps=0, description="",
               poison=True) -> Workload:
    """Build a workload: page table, then q, K and V from their own streams.

    pool_pages defaults to ceil((1 + pool_slack) * pages needed), where pages
    needed counts room for `extra_rows` appended rows per request.
    """
    rng = np.random.default_rng(seed)
    kv_len = np.asarray(kv_len, dtype=np.int64)
    need = int(pages_needed(kv_len + extra_rows, page_size).sum())
    if pool_pages is None:
        pool_pages = max(1, int(math.ceil((1.0 + pool_slack) * need)))
    table = build_page_table(kv_len, page_size, pool_pages, rng)
    B = len(kv_len)
    q = normal((B, num_qo_heads, head_dim), dtype, stream_key(seed, "q"))
    shape = (pool_pages, num_kv_heads, page_size, head_dim)
    k = normal(shape, dtype, stream_key(seed, "k"))
    v = normal(shape, dtype, stream_key(seed, "v"))
    if poison:
        poison_unused(k, v, table, dtype)
    sm_scale = float(np.float32(1.0 / math.sqrt(head_dim)))
    return Workload(name, dtype, num_qo_heads, num_kv_heads, head_dim, table, q, k, v, sm_scale,
                    seed, append_steps, description)


# --- the five workload shapes ---------------------------------------------------------------

def tiny_gqa_f32(seed: int = 1000) -> Workload:
    """batch 1, 8 qo / 2 kv heads, head_dim 64, page 16, kv_len 100 (7 pages, 4 rows
    in the last) drawn from a shuffled pool of 16 pages; f32."""
    return make_paged("tiny_gqa_b1_h8k2_d64_p16_n100_f32", "f32", [100], 8, 2, 64, 16, seed,
                      pool_pages=16, description="tiny paged GQA decode")


def llama3_8b_bf16(seed: int = 1001, batch: int = 32, lo: int = 512, hi: int = 4096) -> Workload:
    """Llama-3-8B-shaped decode layer: 32 qo / 8 kv heads, head_dim 128, page 16,
    kv_len ~ U[512, 4096] per request, pool = need + 10 %; bf16."""
    rng = np.random.default_rng(seed + 7919)
    kv_len = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_paged(f"llama3_8b_b{batch}_h32k8_d128_p16_bf16", "bf16", kv_len, 32, 8, 128, 16,
                      seed, description="Llama-3-8B-shaped decode")


def long_context_f16(seed: int = 1002, batch: int = 4, kv_len: int = 131072) -> Workload:
    """Long-context small batch: 32 qo / 8 kv heads, head_dim 128, page 16,
    kv_len 131072 for every request, pool = need + 10 %; f16."""
    return make_paged(f"longctx_b{batch}_h32k8_d128_p16_n{kv_len}_f16", "f16", [kv_len] * batch,
                      32, 8, 128, 16, seed, description="long-context split-KV decode")


def ragged_70b_bf16(seed: int = 1003, batch: int = 256, max_len: int = 32768) -> Workload:
    """70B-shaped GQA (group 8): 64 qo / 8 kv heads, head_dim 128, page 32,
    kv_len = clip(round(1024 * exp(N(0,1))), 1, max_len) with four forced
    lengths (1, 32, 64, max_len) so kv_len=1, exact page multiples and the
    clip are always present; bf16."""
    rng = np.random.default_rng(seed + 7919)
    kv_len = np.clip(np.rint(1024.0 * np.exp(rng.standard_normal(batch))), 1, max_len).astype(np.int64)
    forced = [1, 32, 64, max_len]
    kv_len[: min(batch, 4)] = forced[: min(batch, 4)]
    return make_paged(f"ragged70b_b{batch}_h64k8_d128_p32_bf16", "bf16", kv_len, 64, 8, 128, 32,
                      seed, description="large ragged batch, group 8")


def mha_append_f16(seed: int = 1004, batch: int = 64, lo: int = 1, hi: int = 8191,
                   steps: int = 8) -> Workload:
    """MHA head_dim 256 with append-then-decode: 16 qo / 16 kv heads, page 16,
    kv_len ~ U[1, 8191], pool with room for `steps` appends + 10 %; f16."""
    rng = np.random.default_rng(seed + 7919)
    kv_len = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_paged(f"mha_d256_append_b{batch}_h16_p16_f16", "f16", kv_len, 16, 16, 256, 16, seed,
                      extra_rows=steps, append_steps=steps, description="MHA d256 append + decode")


CONFIGS = {
    "tiny": tiny_gqa_f32,
    "llama3_8b": llama3_8b_bf16,
    "long_context": long_context_f16,
    "ragged_70b": ragged_70b_bf16,
    "mha_append": mha_append_f16,
}


def contiguous_copy(w: Workload, max_kv_len: int | None = None):
    """The same K/V values laid out as a contiguous [batch, Hk, max_kv_len, D] cache.

    Only valid when every request has the same kv_len (the contiguous entry
    takes one valid_kv_len). Rows past valid_kv_len are NaN.
    """
    t = w.table
    lens = t.kv_len()
    n = int(lens[0])
    if not np.all(lens == n):
        raise ValueError("contiguous copy needs equal kv_len")
    L = max_kv_len or n
    shape = (w.batch, w.num_kv_heads, L, w.head_dim)
    kc = np.full(shape, nan_value(w.dtype), dtype=w.k_data.dtype)
    vc = np.full(shape, nan_value(w.dtype), dtype=w.v_data.dtype)
    P = t.page_size
    for b in range(w.batch):
        pages = t.indices[t.indptr[b]:t.indptr[b + 1]]
        kb = w.k_data[pages].transpose(1, 0, 2, 3).reshape(w.num_kv_heads, len(pages) * P, w.head_dim)
        vb = w.v_data[pages].transpose(1, 0, 2, 3).reshape(w.num_kv_heads, len(pages) * P, w.head_dim)
        kc[b, :, :n] = kb[:, :n]
        vc[b, :, :n] = vb[:, :n]
    return kc, vc, n
