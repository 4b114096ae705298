"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (same library call, same grid planning).
The oracle computes every output; it runs on all host cores."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, compare, to_dev
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
    w = wl.mha_append_f16()
    _append_steps(w, 8, check_pool_every=7)


def test_full_llama3_8b_e4m3_pool():
    """The Llama-3-8B-shaped batch over an E4M3 pool (the benchmark's FP8 configuration)."""
    from tests.test_gpu_fp8 import Fp8Device

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
