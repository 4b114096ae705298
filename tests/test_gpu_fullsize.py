"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (same library call, same grid planning).
The oracle computes every output; it runs on all host cores."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, Fp8Device, compare, to_dev, to_host_raw
from tests.test_gpu_append import _append_steps

pytestmark = pytest.mark.gpu


def test_full_tiny_gqa_f32():
    w = wl.tiny_gqa_f32()
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), "f32", w.name)


def test_full_llama3_8b_bf16():
    w = wl.llama3_8b_bf16()
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), "bf16", w.name)
    assert dw.flags() == 0


def test_full_long_context_f16_paged_and_contiguous():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.long_context_f16()
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    o_ref, lse_ref = oracle.paged_decode_workload(w)
    compare(o, lse, o_ref, lse_ref, "f16", w.name)
    assert dw.flags() == 0
    kc, vc, n = wl.contiguous_copy(w)
    del dw
    kd, vd = to_dev(kc, "f16"), to_dev(vc, "f16")
    qd = to_dev(w.q, "f16")
    o2 = torch.empty_like(qd)
    l2 = torch.empty(w.batch, w.num_qo_heads, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(w.batch, 32, 8, 128, pd.PD_F16))
    pd.pd_contiguous_decode(qd, kd, vd, o2, l2, n, w.sm_scale, ws)
    o_c, lse_c = oracle.contiguous_decode(w.q, kc, vc, w.num_qo_heads, n, w.sm_scale, "f16")
    compare(o2, l2, o_c, lse_c, "f16", w.name + " contiguous")


def test_full_ragged_70b_bf16():
    w = wl.ragged_70b_bf16()
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), "bf16", w.name)
    assert dw.flags() == 0


def test_full_mha_append_f16_eight_steps():
    """Eight steps of pd_paged_append, then pd_paged_decode (the benchmark's
    --append separate step); the whole pool is compared at steps 1 and 8."""
    w = wl.mha_append_f16()
    _append_steps(w, 8, check_pool_every=7)


def test_full_mha_fused_append_decode_eight_steps():
    """Eight steps of pd_paged_append_decode on the full MHA workload (64
    requests, 16 kv heads, head_dim 256, f16): the benchmark's default step for
    it. Every step, the pages that received the new rows are compared bit for
    bit with the oracle's append, and o / lse with the oracle's decode of the
    oracle's pool; the whole K and V pools are compared at steps 1 and 8."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.mha_append_f16()
    dw = DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    t = w.table
    for step in range(w.append_steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        dw.set_table(t)
        pd.pd_paged_append_decode(dw.q, to_dev(kn, "f16"), to_dev(vn, "f16"), dw.k, dw.v, dw.indices, dw.indptr,
                                  dw.lpl, dw.o, dw.lse, w.sm_scale, dw.ws)
        oracle.paged_append(kn, vn, k_host, v_host, t.indices, t.indptr, t.last_page_len, "f16")
        touched = t.indices[t.indptr[1:] - 1]  # each request's last page, where its new row went
        idx = torch.from_numpy(touched.astype(np.int64)).cuda()
        for pool, host, name in ((dw.k, k_host, "K"), (dw.v, v_host, "V")):
            got = pool.view(torch.int16).index_select(0, idx).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, host[touched]), f"{name}: touched pages differ, step {step + 1}"
            if step in (0, w.append_steps - 1):
                assert np.array_equal(to_host_raw(pool, "f16"), host), f"{name}: pool differs, step {step + 1}"
        o_ref, lse_ref = oracle.paged_decode(w.q, k_host, v_host, t.indices, t.indptr, t.last_page_len,
                                             w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size,
                                             w.sm_scale, "f16")
        compare(dw.o, dw.lse, o_ref, lse_ref, "f16", f"fused step {step + 1}")
    assert w.append_steps == 8
    assert dw.flags() == 0


def test_full_llama3_8b_e4m3_pool():
    """The Llama-3-8B-shaped batch over an E4M3 pool (the benchmark's FP8 configuration)."""
    import paged_kv_gqa_13_gb300 as pd

    w = wl.llama3_8b_bf16()
    dev = Fp8Device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", w.name + " e4m3")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_full_long_context_nhd():
    """The long-context batch through the token-major contiguous entry (the benchmark's NHD configuration)."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.long_context_f16()
    kc, vc, n = wl.contiguous_copy(w)
    kc, vc = np.ascontiguousarray(kc.transpose(0, 2, 1, 3)), np.ascontiguousarray(vc.transpose(0, 2, 1, 3))
    kd, vd, qd = to_dev(kc, "f16"), to_dev(vc, "f16"), to_dev(w.q, "f16")
    o = torch.empty_like(qd)
    lse = torch.empty(w.batch, w.num_qo_heads, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(w.batch, 32, 8, 128, pd.PD_F16))
    pd.pd_contiguous_decode_nhd(qd, kd, vd, o, lse, n, w.sm_scale, ws)
    compare(o, lse, *oracle.contiguous_decode(w.q, kc, vc, w.num_qo_heads, n, w.sm_scale, "f16", layout="nhd"),
            "f16", w.name + " nhd")
