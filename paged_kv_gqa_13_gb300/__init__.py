"""pagedecode: batched paged-KV GQA decode attention for sm_103a (GB300).

A thin ctypes binding over the C ABI in ``include/pagedecode.h``
(``libpagedecode.so``, built in-tree by ``build.py``). Each function has the
name of the C entry point it calls and only marshals arguments: every step
of the computation runs in the library's CUDA kernels. Tensors are PyTorch
CUDA tensors (PyTorch supplies device memory and streams); shapes become the
integer arguments of the C call.

The library must be built; importing this package without it raises
ImportError. There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpagedecode.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(
        f"{LIBRARY_PATH} is not built; run `python {os.path.join(_HERE, 'build.py')}` "
        "(needs nvcc with sm_103a support)"
    )

_lib = ctypes.CDLL(LIBRARY_PATH)

PD_F32, PD_F16, PD_BF16 = 0, 1, 2
PD_OK, PD_ERR_INVALID, PD_ERR_UNSUPPORTED, PD_ERR_WORKSPACE, PD_ERR_CUDA = 0, 1, 2, 3, 4
PD_FLAG_BAD_PAGE_ID, PD_FLAG_BAD_LAST_PAGE_LEN, PD_FLAG_BAD_INDPTR, PD_FLAG_WAIT_TIMEOUT = 1, 2, 4, 8
PD_WORKSPACE_HEADER_BYTES = 256
PD_KERNEL_NONE, PD_KERNEL_CUDA_CORES, PD_KERNEL_TENSOR_CORES, PD_KERNEL_FP8_TENSOR_CORES = 0, 1, 2, 3
PD_KERNEL_FP8_TCGEN05 = 4

STATUS_NAMES = {0: "PD_OK", 1: "PD_ERR_INVALID", 2: "PD_ERR_UNSUPPORTED", 3: "PD_ERR_WORKSPACE",
                4: "PD_ERR_CUDA"}

_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_SIGS = {
    "pd_paged_decode_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "pd_paged_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "pd_paged_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _S, _P]),
    "pd_contiguous_decode_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "pd_contiguous_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "pd_merge_states": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _P]),
    "pd_workspace_init": (_I, [_P, _S, _P]),
    "pd_read_device_flags": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "pd_copy_bytes": (_I, [_P, _P, _S, _P]),
    "pd_profile_enable": (_I, [_I]),
    "pd_test_inject_wait_timeout": (_I, [_I]),
    "pd_select_fp8_kernel": (_I, [_I]),
    "pd_profile_read": (_I, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                             ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int),
                             ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    "pd_contiguous_append": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pd_paged_append_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                    _P, _S, _P]),
    "pd_contiguous_append_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "pd_paged_decode_fp8_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "pd_paged_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S,
                                 _P]),
    "pd_paged_append_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _S, _P]),
    "pd_contiguous_decode_nhd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "pd_contiguous_append_nhd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pd_contiguous_append_decode_nhd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S,
                                             _P]),
    "pd_paged_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "pd_paged_decode_noalloc_flags": (_I, [ctypes.POINTER(ctypes.c_int32), _P]),
    "pd_decode_kernel_kind": (_I, [_I, _I, _I, _I, _I]),
    "pd_last_error_string": (ctypes.c_char_p, []),
    "pd_version": (_I, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


class PagedecodeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != PD_OK:
        raise PagedecodeError(status, pd_last_error_string())


def _dtype_code(t) -> int:
    import torch

    codes = {torch.float32: PD_F32, torch.float16: PD_F16, torch.bfloat16: PD_BF16}
    if t.dtype not in codes:
        raise PagedecodeError(PD_ERR_UNSUPPORTED, f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise PagedecodeError(PD_ERR_INVALID, "tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def pd_last_error_string() -> str:
    return _lib.pd_last_error_string().decode()


def pd_version() -> int:
    return _lib.pd_version()


def pd_paged_decode_workspace_bytes(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                                    dtype: int) -> int:
    n = _lib.pd_paged_decode_workspace_bytes(batch, num_qo_heads, num_kv_heads, head_dim, dtype)
    if n == 0:
        raise PagedecodeError(PD_ERR_INVALID, pd_last_error_string())
    return n


def pd_contiguous_decode_workspace_bytes(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                                         dtype: int) -> int:
    n = _lib.pd_contiguous_decode_workspace_bytes(batch, num_qo_heads, num_kv_heads, head_dim, dtype)
    if n == 0:
        raise PagedecodeError(PD_ERR_INVALID, pd_last_error_string())
    return n


def alloc_workspace(nbytes: int, device=None, stream=None):
    """A device byte buffer (256-byte aligned by the allocator) with a zeroed header."""
    import torch

    ws = torch.empty(max(int(nbytes), PD_WORKSPACE_HEADER_BYTES), dtype=torch.uint8, device=device or "cuda")
    pd_workspace_init(ws, stream)
    return ws


def pd_workspace_init(workspace, stream=None) -> None:
    _check(_lib.pd_workspace_init(_ptr(workspace), workspace.numel(), _stream(stream)))


def pd_read_device_flags(workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(_lib.pd_read_device_flags(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return v.value


def pd_paged_decode(q, k_data, v_data, indices, indptr, last_page_len, o, lse, sm_scale: float, workspace,
                    stream=None) -> None:
    """q, o [batch, Hq, D]; k_data, v_data [pages, Hk, page_size, D]; lse [batch, Hq] f32."""
    batch, num_qo_heads, head_dim = q.shape
    num_total_pages, num_kv_heads, page_size, _ = k_data.shape
    _check(_lib.pd_paged_decode(
        _ptr(q), _ptr(k_data), _ptr(v_data), _ptr(indices) if indices.numel() else None, _ptr(indptr),
        _ptr(last_page_len), _ptr(o), _ptr(lse), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
        num_total_pages, indices.numel(), float(sm_scale), _dtype_code(q), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def pd_paged_append_decode(q, k_new, v_new, k_data, v_data, indices, indptr, last_page_len, o, lse,
                           sm_scale: float, workspace, stream=None) -> None:
    """pd_paged_append then pd_paged_decode in one launch; the table already holds the new token."""
    batch, num_qo_heads, head_dim = q.shape
    num_total_pages, num_kv_heads, page_size, _ = k_data.shape
    _check(_lib.pd_paged_append_decode(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_data), _ptr(v_data), _ptr(indices) if indices.numel() else None,
        _ptr(indptr), _ptr(last_page_len), _ptr(o), _ptr(lse), batch, num_qo_heads, num_kv_heads, head_dim,
        page_size, num_total_pages, indices.numel(), float(sm_scale), _dtype_code(q), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def pd_contiguous_append_decode(q, k_new, v_new, k_cache, v_cache, o, lse, position: int, sm_scale: float,
                                workspace, stream=None) -> None:
    """pd_contiguous_append at `position`, then pd_contiguous_decode over position + 1 rows, in one launch."""
    batch, num_qo_heads, head_dim = q.shape
    _, num_kv_heads, max_kv_len, _ = k_cache.shape
    _check(_lib.pd_contiguous_append_decode(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(o),
        _ptr(lse) if lse is not None else None, batch, num_qo_heads, num_kv_heads, head_dim, max_kv_len,
        int(position), float(sm_scale), _dtype_code(q), _ptr(workspace), workspace.numel(), _stream(stream)))


def pd_paged_decode_noalloc(q, k_data, v_data, indices, indptr, last_page_len, o, lse, sm_scale: float,
                            stream=None) -> None:
    """pd_paged_decode with the library's built-in 16 MiB scratch instead of a caller workspace.

    For callers that may not allocate device memory when they call the decode.
    Calls share the scratch: order them on one stream.
    """
    batch, num_qo_heads, head_dim = q.shape
    num_total_pages, num_kv_heads, page_size, _ = k_data.shape
    _check(_lib.pd_paged_decode_noalloc(
        _ptr(q), _ptr(k_data), _ptr(v_data), _ptr(indices) if indices.numel() else None, _ptr(indptr),
        _ptr(last_page_len), _ptr(o), _ptr(lse), batch, num_qo_heads, num_kv_heads, head_dim, page_size,
        num_total_pages, indices.numel(), float(sm_scale), _dtype_code(q), _stream(stream)))


def pd_paged_decode_noalloc_flags(stream=None) -> int:
    """PD_FLAG_* bits set by the last pd_paged_decode_noalloc call on this device (synchronizes the stream)."""
    v = ctypes.c_int32(0)
    _check(_lib.pd_paged_decode_noalloc_flags(ctypes.byref(v), _stream(stream)))
    return v.value


def pd_decode_kernel_kind(num_qo_heads: int, num_kv_heads: int, head_dim: int, dtype: int,
                          fp8_pool: bool = False) -> int:
    """The PD_KERNEL_* a decode of this shape runs (host-side lookup; no device needed)."""
    return _lib.pd_decode_kernel_kind(num_qo_heads, num_kv_heads, head_dim, dtype, 1 if fp8_pool else 0)


def pd_paged_append(k_new, v_new, k_data, v_data, indices, indptr, last_page_len, workspace,
                    stream=None) -> None:
    """k_new, v_new [batch, Hk, D]; the page table is the one after the caller's update."""
    batch, num_kv_heads, head_dim = k_new.shape
    num_total_pages, _, page_size, _ = k_data.shape
    _check(_lib.pd_paged_append(
        _ptr(k_new), _ptr(v_new), _ptr(k_data), _ptr(v_data), _ptr(indices) if indices.numel() else None,
        _ptr(indptr), _ptr(last_page_len), batch, num_kv_heads, head_dim, page_size, num_total_pages,
        indices.numel(), _dtype_code(k_new), _ptr(workspace), workspace.numel(), _stream(stream)))


def pd_contiguous_decode(q, k_cache, v_cache, o, lse, valid_kv_len: int, sm_scale: float, workspace,
                         stream=None) -> None:
    """q, o [batch, Hq, D]; k_cache, v_cache [batch, Hk, max_kv_len, D]; lse [batch, Hq] f32 or None."""
    batch, num_qo_heads, head_dim = q.shape
    _, num_kv_heads, max_kv_len, _ = k_cache.shape
    _check(_lib.pd_contiguous_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), batch, num_qo_heads, num_kv_heads,
        head_dim, max_kv_len, int(valid_kv_len), float(sm_scale), _dtype_code(q), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def pd_merge_states(o_parts, lse_parts, o, lse=None, stream=None) -> None:
    """o_parts [parts, rows, D] f32, lse_parts [parts, rows] f32 (ln) -> o [rows, D], lse [rows]."""
    num_parts, num_rows, head_dim = o_parts.shape
    _check(_lib.pd_merge_states(_ptr(o_parts), _ptr(lse_parts), num_parts, num_rows, head_dim, _ptr(o),
                                _ptr(lse), _dtype_code(o), _stream(stream)))


def pd_copy_bytes(dst, src, nbytes: int | None = None, stream=None) -> None:
    n = nbytes if nbytes is not None else src.numel() * src.element_size()
    _check(_lib.pd_copy_bytes(_ptr(dst), _ptr(src), n, _stream(stream)))


def pd_profile_enable(enable: bool = True) -> None:
    _check(_lib.pd_profile_enable(1 if enable else 0))


def pd_profile_read() -> dict:
    dm, mm, am = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    dn, mn, an = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(_lib.pd_profile_read(ctypes.byref(dm), ctypes.byref(dn), ctypes.byref(mm), ctypes.byref(mn),
                                ctypes.byref(am), ctypes.byref(an)))
    return {"decode_ms": dm.value, "decode_launches": dn.value, "merge_ms": mm.value, "merge_launches": mn.value,
            "append_ms": am.value, "append_launches": an.value}


def pd_contiguous_append(k_new, v_new, k_cache, v_cache, position: int, stream=None) -> None:
    """k_new, v_new [batch, Hk, D] into row `position` of k_cache, v_cache [batch, Hk, max_kv_len, D]."""
    batch, num_kv_heads, head_dim = k_new.shape
    max_kv_len = k_cache.shape[2]
    _check(_lib.pd_contiguous_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), batch, num_kv_heads,
                                     head_dim, max_kv_len, int(position), _dtype_code(k_new), _stream(stream)))


# --- token-major (NHD) contiguous cache: k_cache, v_cache [batch, max_kv_len, Hk, D] ----------

def pd_contiguous_decode_nhd(q, k_cache, v_cache, o, lse, valid_kv_len: int, sm_scale: float, workspace,
                             stream=None) -> None:
    """pd_contiguous_decode on k_cache, v_cache [batch, max_kv_len, Hk, D]."""
    batch, num_qo_heads, head_dim = q.shape
    _, max_kv_len, num_kv_heads, _ = k_cache.shape
    _check(_lib.pd_contiguous_decode_nhd(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), batch, num_qo_heads, num_kv_heads,
        head_dim, max_kv_len, int(valid_kv_len), float(sm_scale), _dtype_code(q), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def pd_contiguous_append_nhd(k_new, v_new, k_cache, v_cache, position: int, stream=None) -> None:
    """k_new, v_new [batch, Hk, D] into token `position` of k_cache, v_cache [batch, max_kv_len, Hk, D]."""
    batch, num_kv_heads, head_dim = k_new.shape
    max_kv_len = k_cache.shape[1]
    _check(_lib.pd_contiguous_append_nhd(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), batch,
                                         num_kv_heads, head_dim, max_kv_len, int(position), _dtype_code(k_new),
                                         _stream(stream)))


def pd_contiguous_append_decode_nhd(q, k_new, v_new, k_cache, v_cache, o, lse, position: int, sm_scale: float,
                                    workspace, stream=None) -> None:
    """pd_contiguous_append_decode on k_cache, v_cache [batch, max_kv_len, Hk, D]."""
    batch, num_qo_heads, head_dim = q.shape
    _, max_kv_len, num_kv_heads, _ = k_cache.shape
    _check(_lib.pd_contiguous_append_decode_nhd(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(o),
        _ptr(lse) if lse is not None else None, batch, num_qo_heads, num_kv_heads, head_dim, max_kv_len,
        int(position), float(sm_scale), _dtype_code(q), _ptr(workspace), workspace.numel(), _stream(stream)))


# --- FP8 (E4M3) pools: k_data, v_data uint8 [pages, Hk, page_size, D]; scales f32 [Hk] ---------

def pd_paged_decode_fp8_workspace_bytes(batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                                        dtype: int) -> int:
    n = _lib.pd_paged_decode_fp8_workspace_bytes(batch, num_qo_heads, num_kv_heads, head_dim, dtype)
    if n == 0:
        raise PagedecodeError(PD_ERR_INVALID, pd_last_error_string())
    return n


def pd_paged_decode_fp8(q, k_data, v_data, k_scale, v_scale, indices, indptr, last_page_len, o, lse,
                        sm_scale: float, workspace, stream=None) -> None:
    """q, o [batch, Hq, D] f16/bf16; k_data, v_data uint8 E4M3 [pages, Hk, page_size, D]; scales f32 [Hk]."""
    batch, num_qo_heads, head_dim = q.shape
    num_total_pages, num_kv_heads, page_size, _ = k_data.shape
    _check(_lib.pd_paged_decode_fp8(
        _ptr(q), _ptr(k_data), _ptr(v_data), _ptr(k_scale), _ptr(v_scale),
        _ptr(indices) if indices.numel() else None, _ptr(indptr), _ptr(last_page_len), _ptr(o), _ptr(lse), batch,
        num_qo_heads, num_kv_heads, head_dim, page_size, num_total_pages, indices.numel(), float(sm_scale),
        _dtype_code(q), _ptr(workspace), workspace.numel(), _stream(stream)))


def pd_paged_append_fp8(k_new, v_new, k_scale, v_scale, k_data, v_data, indices, indptr, last_page_len, workspace,
                        stream=None) -> None:
    """Quantise k_new, v_new [batch, Hk, D] (f16/bf16) into their slots of the E4M3 pools."""
    batch, num_kv_heads, head_dim = k_new.shape
    num_total_pages, _, page_size, _ = k_data.shape
    _check(_lib.pd_paged_append_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(k_scale), _ptr(v_scale), _ptr(k_data), _ptr(v_data),
        _ptr(indices) if indices.numel() else None, _ptr(indptr), _ptr(last_page_len), batch, num_kv_heads,
        head_dim, page_size, num_total_pages, indices.numel(), _dtype_code(k_new), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def pd_select_fp8_kernel(kind: int) -> None:
    """Choose PD_KERNEL_FP8_TENSOR_CORES (default) or PD_KERNEL_FP8_TCGEN05 for E4M3 pools where both apply."""
    _check(_lib.pd_select_fp8_kernel(int(kind)))


def pd_test_inject_wait_timeout(extra_bytes: int) -> None:
    """Test-only: make each decode's first warp wait for bytes that never arrive (0 turns it off)."""
    _check(_lib.pd_test_inject_wait_timeout(int(extra_bytes)))
