"""Shared helpers for the GPU parity tests: device copies of a workload, calls
through the C ABI, and the comparison against the oracle.

Tolerances: o max-abs 1e-5 (f32), 2e-3 (f16), 1.5e-2 (bf16) with V ~ N(0,1);
lse 1e-4 absolute in every dtype; -inf (empty request) must match exactly.
"""
from __future__ import annotations

import numpy as np

O_TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 1.5e-2}
LSE_TOL = 1e-4


def torch_dtype(dtype: str):
    import torch

    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_dev(raw: np.ndarray, dtype: str, device="cuda"):
    """Raw host storage (float32, or uint16 bit patterns) -> CUDA tensor of the dtype."""
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(raw)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(raw).view(np.int16)).to(device)
    return t.view(torch_dtype(dtype))


def to_host_raw(t, dtype: str) -> np.ndarray:
    import torch

    if dtype == "f32":
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def table_dev(table, device="cuda"):
    import torch

    return (torch.from_numpy(table.indices.astype(np.int32)).to(device),
            torch.from_numpy(table.indptr.astype(np.int32)).to(device),
            torch.from_numpy(table.last_page_len.astype(np.int32)).to(device))


class DeviceWorkload:
    """A workload's tensors on the GPU plus output and workspace buffers."""

    def __init__(self, w, device="cuda"):
        import torch

        import paged_kv_gqa_13_gb300 as pd

        self.w = w
        self.q = to_dev(w.q, w.dtype, device)
        self.k = to_dev(w.k_data, w.dtype, device)
        self.v = to_dev(w.v_data, w.dtype, device)
        self.set_table(w.table)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(w.batch, w.num_qo_heads, dtype=torch.float32, device=device)
        code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[w.dtype]
        nbytes = pd.pd_paged_decode_workspace_bytes(w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, code)
        self.ws = pd.alloc_workspace(nbytes, device)

    def set_table(self, table):
        self.table = table
        self.indices, self.indptr, self.lpl = table_dev(table)

    def decode(self):
        import paged_kv_gqa_13_gb300 as pd

        pd.pd_paged_decode(self.q, self.k, self.v, self.indices, self.indptr, self.lpl, self.o, self.lse,
                           self.w.sm_scale, self.ws)
        return self.o, self.lse

    def flags(self) -> int:
        import paged_kv_gqa_13_gb300 as pd

        return pd.pd_read_device_flags(self.ws)


def out_f64(o) -> np.ndarray:
    """Exact float64 values of a float32/float16/bfloat16 CUDA tensor."""
    import torch

    return o.to(torch.float64).cpu().numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype: str, what: str = ""):
    """Assert the tolerances; return (max |do|, max |dlse|)."""
    og = out_f64(o_gpu)
    lg = lse_gpu.double().cpu().numpy() if lse_gpu is not None else None
    assert np.all(np.isfinite(og)), f"{what}: non-finite o"
    do = float(np.max(np.abs(og - o_ref))) if og.size else 0.0
    assert do <= O_TOL[dtype], f"{what}: max |o - o_ref| = {do:.3g} > {O_TOL[dtype]}"
    dl = 0.0
    if lg is not None:
        empty = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), empty), f"{what}: -inf lse mismatch"
        if (~empty).any():
            dl = float(np.max(np.abs(lg[~empty] - lse_ref[~empty])))
        assert dl <= LSE_TOL, f"{what}: max |lse - lse_ref| = {dl:.3g} > {LSE_TOL}"
    return do, dl


class Fp8Device:
    """A workload's E4M3 pool (codes and per-kv-head scales) on the GPU, with outputs and workspace."""

    def __init__(self, w):
        import torch

        import paged_kv_gqa_13_gb300 as pd
        import workloads as wl

        self.w = w
        self.k8, self.v8, self.ks, self.vs = wl.fp8_pool(w)
        self.q = to_dev(w.q, w.dtype)
        self.k = torch.from_numpy(self.k8).cuda()
        self.v = torch.from_numpy(self.v8).cuda()
        self.ksd = torch.from_numpy(self.ks).cuda()
        self.vsd = torch.from_numpy(self.vs).cuda()
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(w.batch, w.num_qo_heads, dtype=torch.float32, device="cuda")
        self.ws = pd.alloc_workspace(pd.pd_paged_decode_fp8_workspace_bytes(
            w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, {"f16": pd.PD_F16, "bf16": pd.PD_BF16}[w.dtype]))
        self.set_table(w.table)

    def set_table(self, t):
        self.t = t
        self.ind, self.ptr, self.lpl = table_dev(t)

    def decode(self):
        import paged_kv_gqa_13_gb300 as pd

        pd.pd_paged_decode_fp8(self.q, self.k, self.v, self.ksd, self.vsd, self.ind, self.ptr, self.lpl, self.o,
                               self.lse, self.w.sm_scale, self.ws)
        return self.o, self.lse

    def oracle_decode(self, k8=None, v8=None):
        import oracle

        t, w = self.t, self.w
        return oracle.paged_decode_fp8(w.q, self.k8 if k8 is None else k8, self.v8 if v8 is None else v8, self.ks,
                                       self.vs, t.indices, t.indptr, t.last_page_len, w.num_qo_heads,
                                       w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale, w.dtype)
