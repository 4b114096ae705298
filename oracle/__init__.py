"""CPU oracle for batched paged-KV decode attention (ctypes binding).

TEST INFRASTRUCTURE ONLY. Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package. The
product library never loads it and it never loads the product library: the
two share no code. The arithmetic lives in ``oracle.cpp`` (plain C++17,
double accumulation, an explicit two-pass softmax over an explicit page-table
walk); this file only builds it and marshals numpy arrays.

Every function is pinned by tests in ``tests/test_oracle.py`` against facts
the problem fixes (closed forms, invariants, brute force), not against
itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_SO = os.path.join(_HERE, "liboracle.so")
# A test that plants a mistake in the oracle points this at a mutant build.
_OVERRIDE = os.environ.get("PD_ORACLE_LIBRARY")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (portable C++17, std::thread)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


_handle = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long


def _lib():
    global _handle
    if _handle is None:
        lib = ctypes.CDLL(_OVERRIDE or build())
        lib.oracle_decode_elements.argtypes = [_P, _I, _L, _P]
        lib.oracle_paged_decode.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _L,
                                            ctypes.c_float, _I, _P, _P, _I]
        lib.oracle_contiguous_decode.argtypes = [_P, _P, _P, _I, _I, _I, _I, _L, _L, ctypes.c_float,
                                                 _I, _I, _P, _P, _I]
        lib.oracle_paged_append.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I]
        lib.oracle_merge_states.argtypes = [_P, _P, _I, _L, _I, _P, _P]
        lib.oracle_contiguous_append.argtypes = [_P, _P, _P, _P, _I, _I, _I, _L, _L, _I, _I]
        lib.oracle_round_to_dtype.argtypes = [_P, _L, _I, _P]
        lib.oracle_paged_decode_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _L,
                                                ctypes.c_float, _I, _P, _P, _I]
        lib.oracle_paged_append_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I]
        lib.oracle_e4m3_values.argtypes = [_P, _L, _P]
        lib.oracle_e4m3_round.argtypes = [_P, _L, _P]
        for f in (lib.oracle_decode_elements, lib.oracle_paged_decode, lib.oracle_contiguous_decode,
                  lib.oracle_paged_append, lib.oracle_merge_states, lib.oracle_round_to_dtype,
                  lib.oracle_contiguous_append, lib.oracle_paged_decode_fp8, lib.oracle_paged_append_fp8,
                  lib.oracle_e4m3_values, lib.oracle_e4m3_round):
            f.restype = _I
        lib.oracle_hardware_threads.restype = _I
        _handle = lib
    return _handle


class OracleError(RuntimeError):
    pass


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def hardware_threads() -> int:
    return int(_lib().oracle_hardware_threads())


def decode_elements(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Exact values of raw storage (float32 array, or uint16 bit patterns) as float64."""
    raw = _c(raw)
    out = np.empty(raw.shape, dtype=np.float64)
    if _lib().oracle_decode_elements(raw.ctypes.data, DTYPE_CODE[dtype], raw.size, out.ctypes.data):
        raise OracleError("decode_elements")
    return out


def paged_decode(q, k_data, v_data, indices, indptr, last_page_len, num_qo_heads, num_kv_heads,
                 head_dim, page_size, sm_scale, dtype, threads: int = 0):
    """o [batch, num_qo_heads, head_dim] and lse [batch, num_qo_heads], float64."""
    q, k_data, v_data = _c(q), _c(k_data), _c(v_data)
    indices = _c(np.asarray(indices), np.int32)
    indptr = _c(np.asarray(indptr), np.int32)
    last_page_len = _c(np.asarray(last_page_len), np.int32)
    batch = len(indptr) - 1
    num_total_pages = k_data.shape[0]
    o = np.empty((batch, num_qo_heads, head_dim), dtype=np.float64)
    lse = np.empty((batch, num_qo_heads), dtype=np.float64)
    rc = _lib().oracle_paged_decode(q.ctypes.data, k_data.ctypes.data, v_data.ctypes.data,
                                    indices.ctypes.data if indices.size else None, indptr.ctypes.data,
                                    last_page_len.ctypes.data, batch, num_qo_heads, num_kv_heads,
                                    head_dim, page_size, num_total_pages, indices.size,
                                    float(sm_scale), DTYPE_CODE[dtype], o.ctypes.data, lse.ctypes.data,
                                    threads)
    if rc:
        raise OracleError(f"oracle_paged_decode returned {rc}")
    return o, lse


def e4m3_values(codes) -> np.ndarray:
    """Exact float64 values of E4M3 codes (uint8 array); NaN for the NaN codes."""
    codes = _c(np.asarray(codes), np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _lib().oracle_e4m3_values(codes.ctypes.data, codes.size, out.ctypes.data)
    return out


def e4m3_round(x) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at +-448."""
    x = _c(np.asarray(x), np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _lib().oracle_e4m3_round(x.ctypes.data, x.size, out.ctypes.data)
    return out


def paged_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, indices, indptr, last_page_len, num_qo_heads,
                     num_kv_heads, head_dim, page_size, sm_scale, q_dtype, threads: int = 0):
    """Decode over an FP8 pool (E4M3 codes, value = code value * scale[kv head]); float64 o, lse."""
    q, k_codes, v_codes = _c(q), _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    k_scale, v_scale = _c(np.asarray(k_scale), np.float32), _c(np.asarray(v_scale), np.float32)
    indices = _c(np.asarray(indices), np.int32)
    indptr = _c(np.asarray(indptr), np.int32)
    last_page_len = _c(np.asarray(last_page_len), np.int32)
    batch = len(indptr) - 1
    o = np.empty((batch, num_qo_heads, head_dim), dtype=np.float64)
    lse = np.empty((batch, num_qo_heads), dtype=np.float64)
    rc = _lib().oracle_paged_decode_fp8(q.ctypes.data, k_codes.ctypes.data, v_codes.ctypes.data,
                                        k_scale.ctypes.data, v_scale.ctypes.data,
                                        indices.ctypes.data if indices.size else None, indptr.ctypes.data,
                                        last_page_len.ctypes.data, batch, num_qo_heads, num_kv_heads, head_dim,
                                        page_size, k_codes.shape[0], indices.size, float(sm_scale),
                                        DTYPE_CODE[q_dtype], o.ctypes.data, lse.ctypes.data, threads)
    if rc:
        raise OracleError(f"oracle_paged_decode_fp8 returned {rc}")
    return o, lse


def paged_append_fp8(k_new, v_new, k_scale, v_scale, k_codes, v_codes, indices, indptr, last_page_len, dtype):
    """Quantise the new rows into the host mirrors k_codes / v_codes (uint8 pools) in place."""
    k_new, v_new = _c(k_new), _c(v_new)
    k_scale, v_scale = _c(np.asarray(k_scale), np.float32), _c(np.asarray(v_scale), np.float32)
    assert k_codes.flags.c_contiguous and v_codes.flags.c_contiguous
    indices = _c(np.asarray(indices), np.int32)
    indptr = _c(np.asarray(indptr), np.int32)
    last_page_len = _c(np.asarray(last_page_len), np.int32)
    num_total_pages, num_kv_heads, page_size, head_dim = k_codes.shape
    rc = _lib().oracle_paged_append_fp8(k_new.ctypes.data, v_new.ctypes.data, k_scale.ctypes.data,
                                        v_scale.ctypes.data, k_codes.ctypes.data, v_codes.ctypes.data,
                                        indices.ctypes.data, indptr.ctypes.data, last_page_len.ctypes.data,
                                        len(indptr) - 1, num_kv_heads, head_dim, page_size, num_total_pages,
                                        DTYPE_CODE[dtype])
    if rc:
        raise OracleError(f"oracle_paged_append_fp8 returned {rc}")


def paged_decode_workload(w, table=None, threads: int = 0):
    """paged_decode on a workloads.Workload (optionally with another table)."""
    t = table or w.table
    return paged_decode(w.q, w.k_data, w.v_data, t.indices, t.indptr, t.last_page_len,
                        w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale,
                        w.dtype, threads)


LAYOUT_CODE = {"hnd": 0, "nhd": 1}


def _contiguous_dims(cache, layout):
    """(batch, num_kv_heads, max_kv_len, head_dim) of an HND [b, Hk, L, D] or NHD [b, L, Hk, D] cache."""
    if layout == "hnd":
        return cache.shape
    batch, max_kv_len, num_kv_heads, head_dim = cache.shape
    return batch, num_kv_heads, max_kv_len, head_dim


def contiguous_decode(q, k_cache, v_cache, num_qo_heads, valid_kv_len, sm_scale, dtype,
                      threads: int = 0, layout: str = "hnd"):
    """q [batch, Hq, D], k/v_cache [batch, Hk, max_kv_len, D] (hnd) or [batch, max_kv_len, Hk, D]
    (nhd); returns float64 o, lse."""
    q, k_cache, v_cache = _c(q), _c(k_cache), _c(v_cache)
    batch, num_kv_heads, max_kv_len, head_dim = _contiguous_dims(k_cache, layout)
    o = np.empty((batch, num_qo_heads, head_dim), dtype=np.float64)
    lse = np.empty((batch, num_qo_heads), dtype=np.float64)
    rc = _lib().oracle_contiguous_decode(q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
                                         batch, num_qo_heads, num_kv_heads, head_dim, max_kv_len,
                                         valid_kv_len, float(sm_scale), DTYPE_CODE[dtype], LAYOUT_CODE[layout],
                                         o.ctypes.data, lse.ctypes.data, threads)
    if rc:
        raise OracleError(f"oracle_contiguous_decode returned {rc}")
    return o, lse


def paged_append(k_new, v_new, k_data, v_data, indices, indptr, last_page_len, dtype):
    """Write the new rows into the host mirrors k_data/v_data in place."""
    k_new, v_new = _c(k_new), _c(v_new)
    assert k_data.flags.c_contiguous and v_data.flags.c_contiguous
    indices = _c(np.asarray(indices), np.int32)
    indptr = _c(np.asarray(indptr), np.int32)
    last_page_len = _c(np.asarray(last_page_len), np.int32)
    num_total_pages, num_kv_heads, page_size, head_dim = k_data.shape
    rc = _lib().oracle_paged_append(k_new.ctypes.data, v_new.ctypes.data, k_data.ctypes.data,
                                    v_data.ctypes.data, indices.ctypes.data, indptr.ctypes.data,
                                    last_page_len.ctypes.data, len(indptr) - 1, num_kv_heads,
                                    head_dim, page_size, num_total_pages, DTYPE_CODE[dtype])
    if rc:
        raise OracleError(f"oracle_paged_append returned {rc}")


def contiguous_append(k_new, v_new, k_cache, v_cache, position, dtype, layout: str = "hnd"):
    """Write token `position` of every (request, kv head) of the host mirrors in place."""
    k_new, v_new = _c(k_new), _c(v_new)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    batch, num_kv_heads, max_kv_len, head_dim = _contiguous_dims(k_cache, layout)
    rc = _lib().oracle_contiguous_append(k_new.ctypes.data, v_new.ctypes.data, k_cache.ctypes.data,
                                         v_cache.ctypes.data, batch, num_kv_heads, head_dim, max_kv_len,
                                         int(position), DTYPE_CODE[dtype], LAYOUT_CODE[layout])
    if rc:
        raise OracleError(f"oracle_contiguous_append returned {rc}")


def merge_states(o_parts, lse_parts):
    """o_parts [parts, rows, D], lse_parts [parts, rows] (float64) -> (o [rows, D], lse [rows])."""
    o_parts = _c(o_parts, np.float64)
    lse_parts = _c(lse_parts, np.float64)
    parts, rows, head_dim = o_parts.shape
    o = np.empty((rows, head_dim), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    if _lib().oracle_merge_states(o_parts.ctypes.data, lse_parts.ctypes.data, parts, rows, head_dim,
                                  o.ctypes.data, lse.ctypes.data):
        raise OracleError("merge_states")
    return o, lse


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """RNE-round float64 values to the storage type; raw storage returned."""
    x = _c(np.asarray(x), np.float64)
    out = np.empty(x.shape, dtype=np.float32 if dtype == "f32" else np.uint16)
    if _lib().oracle_round_to_dtype(x.ctypes.data, x.size, DTYPE_CODE[dtype], out.ctypes.data):
        raise OracleError("round_to_dtype")
    return out
