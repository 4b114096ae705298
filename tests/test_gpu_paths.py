"""GPU parity for paths the workload shapes do not reach: a batch above the
staged page-table size, the contiguous entry on the tensor-core kernel, a long
request split across many units on the tensor-core kernel, and the decode
captured into a CUDA graph and replayed, and outputs in pinned host memory."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hk,dtype", [(16, 4, "bf16"), (16, 2, "f16")])
def test_batch_above_staged_table(hq, hk, dtype):
    # 600 requests: indptr / last_page_len are read from global memory, not staged.
    rng = np.random.default_rng(101)
    lens = rng.integers(0, 70, size=600)
    w = wl.make_paged("big_batch", dtype, lens, hq, hk, 128, 16, seed=102)
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), dtype, "batch 600")
    assert dw.flags() == 0


@pytest.mark.parametrize("dtype,head_dim", [("f16", 128), ("bf16", 64), ("bf16", 256)])
def test_contiguous_on_tensor_cores(dtype, head_dim):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    B, Hq, Hk, L, n = 2, 16, 2, 700, 651  # group 8: the tensor-core kernel
    kc = wl.normal((B, Hk, L, head_dim), dtype, wl.stream_key(110, "k"))
    vc = wl.normal((B, Hk, L, head_dim), dtype, wl.stream_key(110, "v"))
    q = wl.normal((B, Hq, head_dim), dtype, wl.stream_key(110, "q"))
    kc[:, :, n:] = wl.nan_value(dtype)
    vc[:, :, n:] = wl.nan_value(dtype)
    scale = float(np.float32(1 / math.sqrt(head_dim)))
    qd = to_dev(q, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, device="cuda")
    code = pd.PD_F16 if dtype == "f16" else pd.PD_BF16
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, head_dim, code))
    pd.pd_contiguous_decode(qd, to_dev(kc, dtype), to_dev(vc, dtype), o, lse, n, scale, ws)
    compare(o, lse, *oracle.contiguous_decode(q, kc, vc, Hq, n, scale, dtype), dtype, "contiguous mma")


def test_long_request_split_on_tensor_cores():
    w = wl.make_paged("long_mma", "bf16", [40000, 3, 17], 64, 8, 128, 32, seed=111)
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), "bf16", "long request, group 8")


@pytest.mark.parametrize("make", [lambda: wl.llama3_8b_bf16(seed=120, batch=6, lo=100, hi=900),
                                  lambda: wl.ragged_70b_bf16(seed=121, batch=24, max_len=2000)])
def test_decode_replays_from_a_cuda_graph(make):
    # No call of the decode path synchronizes the host, so it can be captured once
    # and replayed; the replay reads the (updated) inputs in place.
    import torch

    w = make()
    dw = DeviceWorkload(w)
    ref_o, ref_lse = (x.clone() for x in dw.decode())  # first call plans the shape
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    dw.o.zero_()
    with torch.cuda.graph(g):
        dw.decode()
    for _ in range(2):
        dw.o.fill_(7)
        dw.lse.fill_(7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dw.o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(dw.lse, ref_lse)
    # new q in place, replay again: matches the oracle on the new input
    q2 = wl.normal(w.q.shape, w.dtype, wl.stream_key(w.seed + 5, "q"))
    dw.q.copy_(to_dev(q2, w.dtype))
    g.replay()
    torch.cuda.synchronize()
    w.q = q2
    compare(dw.o, dw.lse, *oracle.paged_decode_workload(w), w.dtype, "graph replay, new q")


def test_outputs_in_pinned_host_memory():
    """o and lse may be pinned host memory: the decode and merge kernels store
    the results there directly, bit-identical to a device-resident decode."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.llama3_8b_bf16(seed=95, batch=12, lo=1, hi=3000)  # split requests: merged rows and direct rows
    dw = DeviceWorkload(w)
    o_dev, l_dev = [t.clone() for t in dw.decode()]
    oh = torch.empty(o_dev.shape, dtype=o_dev.dtype).pin_memory()
    lh = torch.empty(l_dev.shape, dtype=torch.float32).pin_memory()
    pd.pd_paged_decode(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, oh, lh, w.sm_scale, dw.ws)
    torch.cuda.synchronize()
    assert dw.flags() == 0
    assert torch.equal(oh.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(lh, l_dev.cpu())


def test_copy_bytes_to_and_from_pinned_host_memory():
    """pd_copy_bytes between pinned host memory and device memory, both ways,
    bit for bit, at sizes below, at and above one thread's share of the grid;
    then a decode whose q and page table came in through it matches the
    oracle."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    rng = np.random.default_rng(96)
    for n in (16, 4096, 281_888, 3 << 20):
        h = torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8)).pin_memory()
        d = torch.zeros(n, dtype=torch.uint8, device="cuda")
        pd.pd_copy_bytes(d, h, n)
        back = torch.zeros(n, dtype=torch.uint8).pin_memory()
        pd.pd_copy_bytes(back, d, n)
        torch.cuda.synchronize()
        assert torch.equal(d.cpu(), h), n
        assert torch.equal(back, h), n
    w = wl.llama3_8b_bf16(seed=97, batch=6, lo=1, hi=900)
    dw = DeviceWorkload(w)
    t = w.table
    parts = [np.ascontiguousarray(w.q).view(np.uint8).reshape(-1)] + [
        np.ascontiguousarray(a.astype(np.int32)).view(np.uint8).reshape(-1) for a in (t.indices, t.indptr, t.last_page_len)]
    offs, total = [], 0
    for p in parts:
        offs.append(total)
        total += (p.size + 15) // 16 * 16
    h_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for o_, p in zip(offs, parts):
        h_in[o_:o_ + p.size] = torch.from_numpy(p)
    d_in = torch.zeros(total, dtype=torch.uint8, device="cuda")
    pd.pd_copy_bytes(d_in, h_in, total)
    qd = d_in[offs[0]:offs[0] + parts[0].size].view(dw.q.dtype).view(dw.q.shape)
    ind, ptr, lpl = (d_in[o_:o_ + p.size].view(torch.int32) for o_, p in zip(offs[1:], parts[1:]))
    pd.pd_paged_decode(qd, dw.k, dw.v, ind, ptr, lpl, dw.o, dw.lse, w.sm_scale, dw.ws)
    torch.cuda.synchronize()
    assert dw.flags() == 0
    compare(dw.o, dw.lse, *oracle.paged_decode_workload(w), w.dtype, "inputs copied in by pd_copy_bytes")
