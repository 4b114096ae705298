"""pd_paged_decode_noalloc: the decode for callers that cannot allocate device
memory when they call it (an engine plugin given no scratch, a serving loop
that bans cudaMalloc on its hot path). Its scratch is a static array in the
library. Checked through the C ABI against pd_paged_decode with a caller
workspace, on two calls in a row (the second reuses the array as the first
left it).

This file is named to be collected last, so that a run stopping at its first
failure has run every other test before it.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import LSE_TOL, O_TOL, DeviceWorkload, compare, out_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [
    lambda: wl.llama3_8b_bf16(seed=91, batch=8, lo=300, hi=2500),
    lambda: wl.long_context_f16(seed=92, batch=2, kv_len=9000),
    lambda: wl.make_paged("noalloc_mix", "f16", [0, 1, 16, 700, 33], 16, 16, 256, 16, seed=93),
])
def test_noalloc_matches_workspace_decode_on_two_calls(make):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = make()
    dw = DeviceWorkload(w)
    o_ref, lse_ref = (x.clone() for x in dw.decode())
    for call in range(2):
        o = torch.full_like(dw.o, 9.0)
        lse = torch.full_like(dw.lse, 9.0)
        pd.pd_paged_decode_noalloc(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, o, lse, w.sm_scale)
        torch.cuda.synchronize()
        d_o = float(np.max(np.abs(out_f64(o) - out_f64(o_ref))))
        assert d_o <= O_TOL[w.dtype], f"call {call}: |o - o_workspace| = {d_o}"
        lr, lg = lse_ref.double().cpu().numpy(), lse.double().cpu().numpy()
        empty = np.isneginf(lr)
        assert np.array_equal(np.isneginf(lg), empty)
        if (~empty).any():
            assert float(np.max(np.abs(lg[~empty] - lr[~empty]))) <= LSE_TOL
    # and against the oracle itself
    compare(o, lse, *oracle.paged_decode_workload(w), w.dtype, "noalloc vs oracle")


def test_noalloc_rejects_a_shape_above_its_scratch():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    # 4096 requests x 32 kv heads x 8 heads per tile: the split partials need far more than 16 MiB.
    B, Hq, Hk, D = 4096, 256, 32, 64
    q = torch.zeros(B, Hq, D, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, Hk, 16, D, dtype=torch.float16, device="cuda")
    ind = torch.zeros(0, dtype=torch.int32, device="cuda")
    ptr = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    lpl = torch.zeros(B, dtype=torch.int32, device="cuda")
    lse = torch.zeros(B, Hq, device="cuda")
    with pytest.raises(pd.PagedecodeError) as ei:
        pd.pd_paged_decode_noalloc(q, k, k, ind, ptr, lpl, q, lse, 0.1)
    assert ei.value.status == pd.PD_ERR_WORKSPACE and "16777216" in str(ei.value)


def test_noalloc_flags_are_readable_and_a_rejected_call_enqueues_nothing():
    """The device-side table checks of a noalloc call are read back with
    pd_paged_decode_noalloc_flags. A call that fails its host-side argument
    checks enqueues nothing, not even the clearing of the status word, so the
    previous call's flags are still there after it."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("noalloc_flags", "bf16", [40, 40, 300], 8, 2, 128, 16, seed=94)
    dw = DeviceWorkload(w)
    o_ref, lse_ref = (x.clone() for x in dw.decode())
    o, lse = torch.empty_like(dw.o), torch.empty_like(dw.lse)
    pd.pd_paged_decode_noalloc(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, o, lse, w.sm_scale)
    assert pd.pd_paged_decode_noalloc_flags() == 0
    bad = w.table.copy()
    bad.indices[1] = w.table.num_total_pages + 3  # a page id outside the pool
    dw.set_table(bad)
    pd.pd_paged_decode_noalloc(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, o, lse, w.sm_scale)
    assert pd.pd_paged_decode_noalloc_flags() == pd.PD_FLAG_BAD_PAGE_ID
    with pytest.raises(pd.PagedecodeError) as ei:  # lse missing: rejected on the host
        pd.pd_paged_decode_noalloc(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, o, None, w.sm_scale)
    assert ei.value.status == pd.PD_ERR_INVALID
    assert pd.pd_paged_decode_noalloc_flags() == pd.PD_FLAG_BAD_PAGE_ID
    dw.set_table(w.table)
    pd.pd_paged_decode_noalloc(dw.q, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, o, lse, w.sm_scale)
    assert pd.pd_paged_decode_noalloc_flags() == 0
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(lse, lse_ref)
