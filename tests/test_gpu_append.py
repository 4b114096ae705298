"""GPU parity for pd_paged_append: bit-exact against the oracle's host mirror,
then append-then-decode steps against the oracle."""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, compare, table_dev, to_dev, to_host_raw

pytestmark = pytest.mark.gpu


def _append_steps(w, steps, check_pool_every=1):
    import paged_kv_gqa_13_gb300 as pd

    dw = DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    t = w.table
    for step in range(steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        dw.set_table(t)
        pd.pd_paged_append(to_dev(kn, w.dtype), to_dev(vn, w.dtype), dw.k, dw.v, dw.indices, dw.indptr,
                           dw.lpl, dw.ws)
        oracle.paged_append(kn, vn, k_host, v_host, t.indices, t.indptr, t.last_page_len, w.dtype)
        if step % check_pool_every == 0 or step == steps - 1:
            # bitwise: the pools hold NaN in unused rows
            bits = np.uint32 if w.dtype == "f32" else np.uint16
            assert np.array_equal(to_host_raw(dw.k, w.dtype).view(bits), k_host.view(bits)), f"K differs, step {step}"
            assert np.array_equal(to_host_raw(dw.v, w.dtype).view(bits), v_host.view(bits)), f"V differs, step {step}"
        o, lse = dw.decode()
        o_ref, lse_ref = oracle.paged_decode(w.q, k_host, v_host, t.indices, t.indptr, t.last_page_len,
                                             w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size,
                                             w.sm_scale, w.dtype)
        compare(o, lse, o_ref, lse_ref, w.dtype, f"step {step}")
    assert dw.flags() == 0
    return dw


def test_append_then_decode_mha_d256():
    # Lengths near page boundaries so appends open fresh pages in several steps.
    w = wl.make_paged("append_small", "f16", [15, 16, 1, 31, 47, 200, 3, 64], 16, 16, 256, 16, seed=80,
                      extra_rows=8, append_steps=8)
    _append_steps(w, 8)


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("f32", 64), ("f16", 64)])
def test_append_gqa_shapes(dtype, head_dim):
    w = wl.make_paged(f"append_{dtype}", dtype, [0, 5, 16, 33], 8, 2, head_dim, 16, seed=81, extra_rows=3,
                      append_steps=3)
    _append_steps(w, 3)


def test_append_flags_bad_tables():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("append_bad", "bf16", [5, 5], 8, 2, 128, 16, seed=82, extra_rows=1)
    dw = DeviceWorkload(w)
    kn, vn = w.new_rows(0)
    kd, vd = to_dev(kn, "bf16"), to_dev(vn, "bf16")
    t = wl.table_after_append(w.table)
    t.indices[t.indptr[1] - 1] = -3  # bad page id for request 0
    ind, ptr, lpl = table_dev(t)
    pd.pd_paged_append(kd, vd, dw.k, dw.v, ind, ptr, lpl, dw.ws)
    assert dw.flags() & pd.PD_FLAG_BAD_PAGE_ID
    pd.pd_workspace_init(dw.ws)
    before = dw.k.clone()
    t = wl.table_after_append(w.table)
    t.last_page_len[1] = 0  # slot -1
    ind, ptr, lpl = table_dev(t)
    pd.pd_paged_append(kd, vd, dw.k, dw.v, ind, ptr, lpl, dw.ws)
    assert dw.flags() & pd.PD_FLAG_BAD_LAST_PAGE_LEN
    # in the second call request 0 (good) was written and request 1 was not
    changed = (dw.k.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero()
    assert len(changed) == w.num_kv_heads


# --- contiguous cache ----------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hq,Hk,D,L", [("f16", 32, 8, 128, 300), ("bf16", 64, 8, 128, 97),
                                             ("f32", 8, 8, 64, 40), ("bf16", 16, 4, 256, 65)])
def test_contiguous_append_then_decode(dtype, Hq, Hk, D, L):
    """Each step writes row n of every (request, kv head), bit for bit as the
    oracle does, and a decode over n + 1 rows then matches the oracle."""
    import math

    import torch

    import paged_kv_gqa_13_gb300 as pd

    B, n0, steps = 3, L - 4, 4
    seed = 150 + L
    kc = wl.normal((B, Hk, L, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, Hk, L, D), dtype, wl.stream_key(seed, "v"))
    nan = wl.nan_value(dtype)
    kc[:, :, n0:] = nan
    vc[:, :, n0:] = nan
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(seed, "q"))
    scale = float(np.float32(1 / math.sqrt(D)))
    kd, vd, qd = to_dev(kc, dtype), to_dev(vc, dtype), to_dev(q, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, code))
    bits = np.uint32 if dtype == "f32" else np.uint16
    for step in range(steps):
        n = n0 + step
        kn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "k_new"))
        vn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "v_new"))
        pd.pd_contiguous_append(to_dev(kn, dtype), to_dev(vn, dtype), kd, vd, n)
        oracle.contiguous_append(kn, vn, kc, vc, n, dtype)
        assert np.array_equal(to_host_raw(kd, dtype).view(bits), kc.view(bits)), f"K differs, step {step}"
        assert np.array_equal(to_host_raw(vd, dtype).view(bits), vc.view(bits)), f"V differs, step {step}"
        pd.pd_contiguous_decode(qd, kd, vd, o, lse, n + 1, scale, ws)
        compare(o, lse, *oracle.contiguous_decode(q, kc, vc, Hq, n + 1, scale, dtype), dtype, f"step {step}")
    assert pd.pd_read_device_flags(ws) == 0


def test_contiguous_append_rejects_position_past_the_cache():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    kn = torch.zeros(2, 2, 64, dtype=torch.float16, device="cuda")
    kc = torch.zeros(2, 2, 10, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(pd.PagedecodeError):
        pd.pd_contiguous_append(kn, kn, kc, kc, 10)
    assert torch.all(kc == 0)


# --- append fused into the decode launch ---------------------------------------------------

@pytest.mark.parametrize("dtype,Hq,Hk,D", [
    ("f16", 16, 16, 256),   # MHA, CUDA cores
    ("bf16", 32, 8, 128),   # group 4, tensor cores
    ("bf16", 64, 8, 128),   # group 8, tensor cores
    ("bf16", 32, 2, 128),   # group 16: two head tiles write the same row, tensor cores
    ("f32", 24, 2, 64),     # group 12: two head tiles of 6, CUDA cores
    ("f16", 8, 8, 64),
])
def test_fused_append_decode(dtype, Hq, Hk, D):
    """Per step, pd_paged_append_decode leaves the pool bit for bit as the
    oracle's append does and decodes it as the oracle does; o and lse are
    also bit-identical to pd_paged_append followed by pd_paged_decode."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    steps = 5
    # a request that starts empty, page-boundary lengths, and one long enough to be split
    w = wl.make_paged(f"fused_{dtype}_{Hq}_{Hk}", dtype, [0, 15, 16, 1, 31, 2500, 3, 64], Hq, Hk, D, 16,
                      seed=170 + Hq + Hk, extra_rows=steps, append_steps=steps)
    fused = DeviceWorkload(w)
    split = DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    bits = np.uint32 if dtype == "f32" else np.uint16
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
        assert np.array_equal(to_host_raw(fused.k, dtype).view(bits), k_host.view(bits)), f"K differs, step {step}"
        assert np.array_equal(to_host_raw(fused.v, dtype).view(bits), v_host.view(bits)), f"V differs, step {step}"
        o_ref, lse_ref = oracle.paged_decode(w.q, k_host, v_host, t.indices, t.indptr, t.last_page_len,
                                             w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size,
                                             w.sm_scale, dtype)
        compare(fused.o, fused.lse, o_ref, lse_ref, dtype, f"fused step {step}")
        raw = (lambda x: x) if dtype == "f32" else (lambda x: x.view(torch.int16))
        assert torch.equal(raw(fused.o), raw(o2)), f"fused o differs from append + decode, step {step}"
        assert torch.equal(fused.lse, l2), f"fused lse differs from append + decode, step {step}"
    assert fused.flags() == 0 and split.flags() == 0


def test_fused_append_decode_flags_bad_tables():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("fused_bad", "bf16", [5, 5, 9], 8, 2, 128, 16, seed=183, extra_rows=1)
    dw = DeviceWorkload(w)
    kn, vn = w.new_rows(0)
    kd, vd = to_dev(kn, "bf16"), to_dev(vn, "bf16")
    before = dw.k.clone()
    t = wl.table_after_append(w.table)
    t.last_page_len[1] = 0  # request 1: no row to write into
    dw.set_table(t)
    pd.pd_paged_append_decode(dw.q, kd, vd, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, dw.o, dw.lse,
                              w.sm_scale, dw.ws)
    assert dw.flags() & pd.PD_FLAG_BAD_LAST_PAGE_LEN
    changed = (dw.k.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero()
    assert len(changed) == 2 * w.num_kv_heads  # requests 0 and 2 only
    # a request with no page at all cannot take the new token
    pd.pd_workspace_init(dw.ws)
    t = wl.table_after_append(w.table)
    # request 1 loses its pages
    t2 = dataclasses.replace(
        t, indices=np.concatenate([t.indices[:t.indptr[1]], t.indices[t.indptr[2]:]]),
        indptr=np.array([0, t.indptr[1], t.indptr[1], t.indptr[1] + t.indptr[3] - t.indptr[2]], dtype=t.indptr.dtype))
    dw.set_table(t2)
    pd.pd_paged_append_decode(dw.q, kd, vd, dw.k, dw.v, dw.indices, dw.indptr, dw.lpl, dw.o, dw.lse,
                              w.sm_scale, dw.ws)
    assert dw.flags() & pd.PD_FLAG_BAD_INDPTR
    assert torch.all(torch.isneginf(dw.lse[1])) and torch.all(dw.o[1].float() == 0)


@pytest.mark.parametrize("dtype,Hq,Hk,D,L", [("f16", 32, 8, 128, 300), ("bf16", 64, 8, 128, 97),
                                             ("f32", 8, 8, 64, 40)])
def test_fused_contiguous_append_decode(dtype, Hq, Hk, D, L):
    import math

    import torch

    import paged_kv_gqa_13_gb300 as pd

    B, n0, steps = 3, L - 4, 4
    seed = 190 + L
    kc = wl.normal((B, Hk, L, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, Hk, L, D), dtype, wl.stream_key(seed, "v"))
    nan = wl.nan_value(dtype)
    kc[:, :, n0:] = nan
    vc[:, :, n0:] = nan
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(seed, "q"))
    scale = float(np.float32(1 / math.sqrt(D)))
    kd, vd, qd = to_dev(kc, dtype), to_dev(vc, dtype), to_dev(q, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, code))
    bits = np.uint32 if dtype == "f32" else np.uint16
    for step in range(steps):
        n = n0 + step
        kn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "k_new"))
        vn = wl.normal((B, Hk, D), dtype, wl.stream_key(seed + step, "v_new"))
        pd.pd_contiguous_append_decode(qd, to_dev(kn, dtype), to_dev(vn, dtype), kd, vd, o, lse, n, scale, ws)
        oracle.contiguous_append(kn, vn, kc, vc, n, dtype)
        assert np.array_equal(to_host_raw(kd, dtype).view(bits), kc.view(bits)), f"K differs, step {step}"
        assert np.array_equal(to_host_raw(vd, dtype).view(bits), vc.view(bits)), f"V differs, step {step}"
        compare(o, lse, *oracle.contiguous_decode(q, kc, vc, Hq, n + 1, scale, dtype), dtype, f"step {step}")
    assert pd.pd_read_device_flags(ws) == 0
