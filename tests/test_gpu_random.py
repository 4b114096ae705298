"""Randomised GPU parity sweep: seeded random shapes, tables and lengths across
every decode path, each output against the CPU oracle.

Each case draws, from its own seed: the dtype, head_dim, q / kv head counts
(groups 1..16, so every kernel and head-tile split is reached), the page size
(1..128 rows), the batch (up to 600, past the 512 requests whose table is
staged in shared memory) and ragged lengths (empty, one row, page multiples and
a lognormal body up to ~20,000 rows). Some tables also list page ids that no
request uses before and after the requests' ranges. The cases are fixed by
their seeds, so a failure reproduces.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, Fp8Device, compare, to_dev, to_host_raw

pytestmark = pytest.mark.gpu

GROUPS = [(1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (6, 1), (8, 1), (12, 1), (16, 1)]


def draw_case(seed: int):
    rng = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][int(rng.integers(3))]
    head_dim = [64, 128, 256][int(rng.integers(3))]
    g, _ = GROUPS[int(rng.integers(len(GROUPS)))]
    hk = int(rng.choice([1, 2, 4, 8]))
    page = int(rng.choice([1, 3, 8, 16, 16, 16, 32, 48, 100, 128]))
    batch = int(rng.choice([1, 3, 17, 64, 130, 513, 600]))
    # lengths: a lognormal body plus forced special values
    body = np.clip(np.rint(np.exp(rng.normal(np.log(300), 1.3, size=batch))), 0, 20000).astype(np.int64)
    forced = [0, 1, page, 2 * page, 3 * page + 1]
    body[: min(batch, len(forced))] = forced[: min(batch, len(forced))]
    # keep the oracle's work bounded: ~3e5 rows in total
    while body.sum() * hk > 300_000:
        body = body // 2
    rng.shuffle(body)
    return dtype, head_dim, g * hk, hk, page, body


def with_unlisted_entries(w, lead: int, trail: int):
    """The same table with `lead` and `trail` unused page ids listed around the requests' ranges."""
    import dataclasses

    t = w.table
    spare = t.free_pages[: max(lead, trail)] if t.free_pages else []
    if len(spare) < max(lead, trail):
        return t
    ind = np.concatenate([np.asarray(spare[:lead], np.int32), t.indices, np.asarray(spare[:trail], np.int32)])
    return dataclasses.replace(t, indices=ind.astype(np.int32), indptr=(t.indptr + lead).astype(np.int32))


@pytest.mark.parametrize("seed", list(range(1000, 1120)))
def test_random_paged_decode(seed):
    dtype, D, hq, hk, page, lens = draw_case(seed)
    w = wl.make_paged(f"rand{seed}", dtype, lens, hq, hk, D, page, seed=seed, pool_slack=0.2)
    t = with_unlisted_entries(w, int(seed % 3), int(seed % 5)) if seed % 2 else w.table
    dw = DeviceWorkload(w)
    dw.set_table(t)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w, table=t), dtype,
            f"seed {seed}: {dtype} D{D} {hq}/{hk} page {page} batch {len(lens)}")
    assert dw.flags() == 0


@pytest.mark.parametrize("seed", list(range(2000, 2024)))
def test_random_fused_append_decode(seed):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    dtype, D, hq, hk, page, lens = draw_case(seed)
    steps = 2
    w = wl.make_paged(f"randapp{seed}", dtype, lens, hq, hk, D, page, seed=seed, extra_rows=steps,
                      append_steps=steps)
    dw = DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    bits = np.uint32 if dtype == "f32" else np.uint16
    t = w.table
    for step in range(steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        dw.set_table(t)
        pd.pd_paged_append_decode(dw.q, to_dev(kn, dtype), to_dev(vn, dtype), dw.k, dw.v, dw.indices, dw.indptr,
                                  dw.lpl, dw.o, dw.lse, w.sm_scale, dw.ws)
        oracle.paged_append(kn, vn, k_host, v_host, t.indices, t.indptr, t.last_page_len, dtype)
        assert np.array_equal(to_host_raw(dw.k, dtype).view(bits), k_host.view(bits)), f"seed {seed}: K pool"
        assert np.array_equal(to_host_raw(dw.v, dtype).view(bits), v_host.view(bits)), f"seed {seed}: V pool"
        o_ref, lse_ref = oracle.paged_decode(w.q, k_host, v_host, t.indices, t.indptr, t.last_page_len,
                                             hq, hk, D, page, w.sm_scale, dtype)
        compare(dw.o, dw.lse, o_ref, lse_ref, dtype, f"seed {seed} step {step}")
    assert dw.flags() == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("seed", list(range(3000, 3020)))
def test_random_contiguous_decode(seed):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    rng = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][int(rng.integers(3))]
    D = [64, 128, 256][int(rng.integers(3))]
    g, _ = GROUPS[int(rng.integers(len(GROUPS)))]
    hk = int(rng.choice([1, 2, 8]))
    hq = g * hk
    B = int(rng.integers(1, 6))
    L = int(rng.integers(1, 6000 // hk))
    valid = int(rng.integers(0, L + 1))
    kc = wl.normal((B, hk, L, D), dtype, wl.stream_key(seed, "k"))
    vc = wl.normal((B, hk, L, D), dtype, wl.stream_key(seed, "v"))
    kc[:, :, valid:] = wl.nan_value(dtype)
    vc[:, :, valid:] = wl.nan_value(dtype)
    q = wl.normal((B, hq, D), dtype, wl.stream_key(seed, "q"))
    scale = float(np.float32(1 / math.sqrt(D)))
    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, hq, hk, D, code))
    qd = to_dev(q, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, hq, dtype=torch.float32, device="cuda")
    nhd = bool(seed % 2)
    if nhd:
        kt, vt = np.ascontiguousarray(kc.transpose(0, 2, 1, 3)), np.ascontiguousarray(vc.transpose(0, 2, 1, 3))
        pd.pd_contiguous_decode_nhd(qd, to_dev(kt, dtype), to_dev(vt, dtype), o, lse, valid, scale, ws)
        ref = oracle.contiguous_decode(q, kt, vt, hq, valid, scale, dtype, layout="nhd")
    else:
        pd.pd_contiguous_decode(qd, to_dev(kc, dtype), to_dev(vc, dtype), o, lse, valid, scale, ws)
        ref = oracle.contiguous_decode(q, kc, vc, hq, valid, scale, dtype)
    compare(o, lse, *ref, dtype, f"seed {seed}: {dtype} D{D} {hq}/{hk} B{B} L{L} valid {valid} nhd {nhd}")
    assert pd.pd_read_device_flags(ws) == 0


@pytest.mark.parametrize("seed", list(range(4000, 4020)))
def test_random_e4m3_decode(seed):
    import paged_kv_gqa_13_gb300 as pd

    dtype, D, hq, hk, page, lens = draw_case(seed)
    if dtype == "f32":
        dtype = "bf16"
    w = wl.make_paged(f"rande4m3{seed}", dtype, lens, hq, hk, D, page, seed=seed)
    dev = Fp8Device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), dtype, f"seed {seed}: e4m3 {dtype} D{D} {hq}/{hk} page {page}")
    assert pd.pd_read_device_flags(dev.ws) == 0
