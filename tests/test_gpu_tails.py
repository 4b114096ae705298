"""Dynamic share tails of the decode kernels: shapes with enough positions
per warp that the last eighth of each warp's share is handed out at run time to
the warps that finish first. The unit boundaries are fixed, so the results must
not depend on which warp ran which tail, and the tail counters in the workspace
header must be back at zero after every call."""
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, compare

pytestmark = pytest.mark.gpu

TAIL_CTL = 64  # workspace header bytes of the two tail counters


def _counters(ws):
    import torch

    return ws[TAIL_CTL:TAIL_CTL + 8].view(torch.int32).cpu().tolist()


@pytest.mark.parametrize("make", [
    # Llama-shaped, ~30 positions (pages x kv heads) per warp
    lambda: wl.llama3_8b_bf16(seed=71, batch=24, lo=2000, hi=4096),
    # group 8, mixed lengths with empty-ish requests, ~22 positions per warp
    lambda: wl.make_paged("tails_f16_g8", "f16", [20000, 1, 8000, 17, 24000, 600], 64, 8, 128, 16, seed=72),
    # one-row pages at head_dim 64: ~50 positions per warp, segments of over 32 parts
    lambda: wl.make_paged("tails_bf16_d64_p1", "bf16", [3000, 5000, 1], 32, 8, 64, 1, seed=73),
    # f32 MHA on the CUDA-core kernel, ~16 positions per warp
    lambda: wl.make_paged("tails_f32_mha", "f32", [12000, 1, 9000, 17, 10000], 8, 8, 128, 16, seed=76),
])
def test_tails_repeatable_and_match_oracle(make):
    import torch

    w = make()
    dw = DeviceWorkload(w)
    o1, l1 = [t.clone() for t in dw.decode()]
    assert dw.flags() == 0
    assert _counters(dw.ws) == [0, 0]
    for _ in range(3):
        o, lse = dw.decode()
        assert torch.equal(o, o1) if w.dtype == "f32" else torch.equal(o.view(torch.int16), o1.view(torch.int16))
        assert torch.equal(lse, l1)
    assert _counters(dw.ws) == [0, 0]
    compare(o1, l1, *oracle.paged_decode_workload(w), w.dtype, "tails")


def test_tails_on_the_token_major_cache():
    """NHD contiguous cache with 8 kv heads (the per-token-range unit layout),
    ~50 positions per warp: tails taken at run time, results repeatable bit for
    bit and equal to the oracle's."""
    import math

    import numpy as np
    import torch

    import paged_kv_gqa_13_gb300 as pd
    from tests.gpu_helpers import to_dev

    B, L, valid, Hq, Hk, D, dtype = 3, 40000, 39990, 32, 8, 128, "f16"
    seed = 75
    kc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, L, Hk, D), dtype, wl.stream_key(seed, "v"))
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(seed, "q"))
    kc[:, valid:] = wl.nan_value(dtype)
    vc[:, valid:] = wl.nan_value(dtype)
    scale = float(np.float32(1 / math.sqrt(D)))
    qd, kd, vd = to_dev(q, dtype), to_dev(kc, dtype), to_dev(vc, dtype)
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, pd.PD_F16))
    o1 = torch.empty_like(qd)
    l1 = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    pd.pd_contiguous_decode_nhd(qd, kd, vd, o1, l1, valid, scale, ws)
    assert pd.pd_read_device_flags(ws) == 0
    for _ in range(3):
        o = torch.empty_like(qd)
        lse = torch.empty_like(l1)
        pd.pd_contiguous_decode_nhd(qd, kd, vd, o, lse, valid, scale, ws)
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, l1)
    assert _counters(ws) == [0, 0]
    o_ref, lse_ref = oracle.contiguous_decode(q, kc, vc, Hq, valid, scale, dtype, layout="nhd")
    compare(o1, l1, o_ref, lse_ref, dtype, "nhd with tails")


@pytest.mark.parametrize("dtype,Hq,Hk,D,lens", [
    ("bf16", 32, 8, 128, [20000, 0, 15, 9000, 16000, 1]),   # tensor cores, ~19 positions per warp
    ("f16", 16, 16, 256, [12000, 1, 7000]),                 # CUDA cores (MHA), ~16 positions per warp
])
def test_tails_with_the_fused_append(dtype, Hq, Hk, D, lens):
    """Fused append + decode on shapes that take tails: the pool ends bit for
    bit as the oracle's append leaves it, o and lse are bit-identical to the
    append launch followed by the decode, and they match the oracle."""
    import numpy as np
    import torch

    import paged_kv_gqa_13_gb300 as pd
    from tests.gpu_helpers import to_dev, to_host_raw

    steps = 2
    w = wl.make_paged(f"tails_fused_{dtype}_{Hq}_{Hk}", dtype, lens, Hq, Hk, D, 16, seed=77 + Hq,
                      extra_rows=steps, append_steps=steps)
    fused, split = DeviceWorkload(w), DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    t = w.table
    for step in range(steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        knd, vnd = to_dev(kn, dtype), to_dev(vn, dtype)
        fused.set_table(t)
        split.set_table(t)
        pd.pd_paged_append_decode(fused.q, knd, vnd, fused.k, fused.v, fused.indices, fused.indptr, fused.lpl,
                                  fused.o, fused.lse, w.sm_scale, fused.ws)
        pd.pd_paged_append(knd, vnd, split.k, split.v, split.indices, split.indptr, split.lpl, split.ws)
        o2, l2 = split.decode()
        oracle.paged_append(kn, vn, k_host, v_host, t.indices, t.indptr, t.last_page_len, dtype)
        assert np.array_equal(to_host_raw(fused.k, dtype).view(np.uint16), k_host.view(np.uint16))
        assert np.array_equal(to_host_raw(fused.v, dtype).view(np.uint16), v_host.view(np.uint16))
        assert torch.equal(fused.o.view(torch.int16), o2.view(torch.int16)) and torch.equal(fused.lse, l2)
        assert fused.flags() == 0 and split.flags() == 0
        assert _counters(fused.ws) == [0, 0] and _counters(split.ws) == [0, 0]
        o_ref, lse_ref = oracle.paged_decode(w.q, k_host, v_host, t.indices, t.indptr, t.last_page_len,
                                             w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale,
                                             dtype)
        compare(fused.o, fused.lse, o_ref, lse_ref, dtype, f"fused with tails, step {step}")
