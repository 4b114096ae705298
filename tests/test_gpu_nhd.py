"""GPU parity for the token-major (NHD) contiguous cache, [batch, max_kv_len, Hk, D]:
decode against the oracle and against the HND entry on the transposed cache;
append and fused append + decode bit-exact against the oracle."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import LSE_TOL, O_TOL, compare, to_dev, to_host_raw

pytestmark = pytest.mark.gpu

CODE = {"f32": 0, "f16": 1, "bf16": 2}


def _raw(t, dtype):
    import torch

    return t if dtype == "f32" else t.view(torch.int16)


@pytest.mark.parametrize("dtype,Hq,Hk,D,L,valid", [
    ("f16", 32, 8, 128, 5000, 4999),   # group 4, tensor cores, per-token-range units
    ("bf16", 64, 8, 128, 777, 700),    # group 8, tensor cores
    ("bf16", 16, 2, 256, 300, 291),    # group 8, D 256, tensor cores
    ("f32", 8, 8, 64, 100, 100),       # MHA f32
    ("f16", 16, 16, 256, 90, 33),      # MHA D 256
    ("f32", 24, 2, 128, 64, 1),        # group 12: two head tiles
    ("f16", 32, 4, 64, 20000, 19999),  # long, D 64
])
def test_nhd_decode_matches_oracle_and_hnd(dtype, Hq, Hk, D, L, valid):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    B = 3
    seed = 200 + L + Hq
    kc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "v"))
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(seed, "q"))
    nan = wl.nan_value(dtype)
    kc[:, valid:] = nan
    vc[:, valid:] = nan
    scale = float(np.float32(1 / math.sqrt(D)))
    o_ref, lse_ref = oracle.contiguous_decode(q, kc, vc, Hq, valid, scale, dtype, layout="nhd")
    qd, kd, vd = to_dev(q, dtype), to_dev(kc, dtype), to_dev(vc, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, CODE[dtype]))
    pd.pd_contiguous_decode_nhd(qd, kd, vd, o, lse, valid, scale, ws)
    compare(o, lse, o_ref, lse_ref, dtype, "nhd")
    # The same values in HND order. When the passes fill a block's warps the
    # NHD entry lays its units out per token range, so requests split at other
    # points than in HND order and partial sums round differently: equal within
    # the tolerance, and bit-identical across repeated NHD calls.
    o2 = torch.empty_like(qd)
    l2 = torch.empty_like(lse)
    pd.pd_contiguous_decode(qd, kd.transpose(1, 2).contiguous(), vd.transpose(1, 2).contiguous(), o2, l2, valid,
                            scale, ws)
    assert float((o.double() - o2.double()).abs().max()) <= 2 * O_TOL[dtype]
    assert float((lse.double() - l2.double()).abs().max()) <= 2 * LSE_TOL
    o3 = torch.empty_like(qd)
    l3 = torch.empty_like(lse)
    pd.pd_contiguous_decode_nhd(qd, kd, vd, o3, l3, valid, scale, ws)
    assert torch.equal(_raw(o, dtype), _raw(o3, dtype)) and torch.equal(lse, l3)
    assert pd.pd_read_device_flags(ws) == 0


def test_nhd_zero_valid_rows():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    q = torch.randn(2, 8, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(2, 10, 2, 64, device="cuda", dtype=torch.bfloat16)
    o = torch.full_like(q, 7.0)
    lse = torch.zeros(2, 8, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(2, 8, 2, 64, pd.PD_BF16))
    pd.pd_contiguous_decode_nhd(q, k, k, o, lse, 0, 0.125, ws)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("dtype,Hq,Hk,D,L", [("f16", 32, 8, 128, 300), ("bf16", 64, 8, 128, 97),
                                             ("f32", 8, 8, 64, 40), ("bf16", 16, 4, 256, 65),
                                             ("f16", 32, 8, 128, 40000)])  # ~50 positions per warp: share tails
def test_nhd_append_then_decode(dtype, Hq, Hk, D, L, fused):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    B, n0, steps = 3, L - 4, 4
    seed = 230 + L
    kc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "v"))
    nan = wl.nan_value(dtype)
    kc[:, n0:] = nan
    vc[:, n0:] = nan
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(seed, "q"))
    scale = float(np.float32(1 / math.sqrt(D)))
    kd, vd, qd = to_dev(kc, dtype), to_dev(vc, dtype), to_dev(q, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, CODE[dtype]))
    bits = np.uint32 if dtype == "f32" else np.uint16
    for step in range(steps):
        n = n0 + step
        kn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "k_new"))
        vn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "v_new"))
        knd, vnd = to_dev(kn, dtype), to_dev(vn, dtype)
        if fused:
            pd.pd_contiguous_append_decode_nhd(qd, knd, vnd, kd, vd, o, lse, n, scale, ws)
        else:
            pd.pd_contiguous_append_nhd(knd, vnd, kd, vd, n)
            pd.pd_contiguous_decode_nhd(qd, kd, vd, o, lse, n + 1, scale, ws)
        oracle.contiguous_append(kn, vn, kc, vc, n, dtype, layout="nhd")
        assert np.array_equal(to_host_raw(kd, dtype).view(bits), kc.view(bits)), f"K differs, step {step}"
        assert np.array_equal(to_host_raw(vd, dtype).view(bits), vc.view(bits)), f"V differs, step {step}"
        compare(o, lse, *oracle.contiguous_decode(q, kc, vc, Hq, n + 1, scale, dtype, layout="nhd"), dtype,
                f"step {step}")
    assert pd.pd_read_device_flags(ws) == 0
