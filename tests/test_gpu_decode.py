"""GPU parity: pd_paged_decode / pd_contiguous_decode / pd_merge_states through
the C ABI against the CPU oracle on the same seeded bytes."""
import math
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, LSE_TOL, O_TOL, compare, out_f64, to_dev

pytestmark = pytest.mark.gpu


def _run(w, threads=0):
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    o_ref, lse_ref = oracle.paged_decode_workload(w, threads=threads)
    err = compare(o, lse, o_ref, lse_ref, w.dtype, w.name)
    assert dw.flags() == 0
    return dw, err


# --- the five workload shapes at sizes the oracle finishes in seconds -----------------------

def test_tiny_gqa_f32_full_size():
    _run(wl.tiny_gqa_f32())


def test_llama3_8b_shape_small_batch():
    _run(wl.llama3_8b_bf16(seed=11, batch=6, lo=512, hi=1500))


def test_long_context_shape_split_over_many_warps():
    # 4 requests x 8 kv heads over ~1200 warps: every request is split.
    _run(wl.long_context_f16(seed=12, batch=4, kv_len=20000 + 7))


def test_ragged_70b_shape_group8():
    _run(wl.ragged_70b_bf16(seed=13, batch=40, max_len=6000))


def test_mha_d256_shape():
    _run(wl.mha_append_f16(seed=14, batch=12, lo=1, hi=2000, steps=0))


# --- every supported (dtype, head_dim, group) combination, ragged lengths --------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("hq,hk", [(4, 4), (8, 4), (8, 2), (16, 2), (6, 2), (12, 1), (16, 1)])
def test_dtype_headdim_group_grid(dtype, head_dim, hq, hk):
    rng = np.random.default_rng(zlib.crc32(f"{dtype}/{head_dim}/{hq}/{hk}".encode()))
    lens = rng.integers(1, 300, size=5)
    lens[0] = 1
    w = wl.make_paged(f"grid_{dtype}_{head_dim}_{hq}_{hk}", dtype, lens, hq, hk, head_dim, 16,
                      seed=int(rng.integers(1 << 30)))
    _run(w)


@pytest.mark.parametrize("page_size", [1, 8, 16, 32, 64, 100])
@pytest.mark.parametrize("hq,hk,dtype", [(16, 4, "bf16"), (16, 2, "bf16"), (16, 2, "f16")])
def test_page_sizes(page_size, hq, hk, dtype):
    # Groups 4 and 8 in 16 bits both run on the tensor-core kernel (16-row TMA
    # boxes); the CUDA-core kernel's page sizes are in test_gpu_cuda_core_pages.py.
    import paged_kv_gqa_13_gb300 as pd

    assert pd.pd_decode_kernel_kind(hq, hk, 128, {"f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]) == \
        pd.PD_KERNEL_TENSOR_CORES
    w = wl.make_paged(f"pages_{page_size}", dtype, [1, page_size, 2 * page_size, 333, 50, 17], hq, hk, 128,
                      page_size, seed=40 + page_size)
    _run(w)


# --- page-table special cases --------------------------------------------------------------

def test_empty_requests_and_zero_length_last_page():
    import torch

    w = wl.make_paged("empties", "f16", [0, 40, 0, 16, 5], 8, 2, 128, 16, seed=50)
    t = w.table.copy()
    # request 3 (16 rows, one full page) gets an extra page with 0 valid rows
    extra = t.free_pages[0]
    ind = list(t.indices)
    ind.insert(int(t.indptr[4]), extra)
    t.indices = np.asarray(ind, dtype=np.int32)
    t.indptr[4:] += 1
    t.last_page_len[3] = 0
    dw = DeviceWorkload(w)
    dw.set_table(t)
    o, lse = dw.decode()
    o_ref, lse_ref = oracle.paged_decode_workload(w, table=t)
    compare(o, lse, o_ref, lse_ref, "f16", "empties")
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    assert dw.flags() == 0


def test_all_requests_empty():
    w = wl.make_paged("all_empty", "bf16", [0, 0, 0], 8, 2, 64, 16, seed=51, pool_pages=4)
    dw, _ = _run(w)


def test_kv_len_one_returns_the_v_row_exactly():
    w = wl.make_paged("len1", "bf16", [1] * 7, 32, 8, 128, 16, seed=52)
    dw, _ = _run(w)
    t = w.table
    g = w.group
    for b in range(w.batch):
        page = t.indices[t.indptr[b]]
        for h in range(w.num_qo_heads):
            assert np.array_equal(out_f64(dw.o[b, h]), oracle.decode_elements(w.v_data[page, h // g, 0], "bf16"))


def test_one_long_request_among_short_ones():
    w = wl.make_paged("skew", "bf16", [30000, 1, 2, 17, 3, 64], 32, 8, 128, 16, seed=53)
    _run(w)


def test_bad_page_id_and_last_page_len_are_flagged_not_fatal():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("bad", "f16", [40, 40], 8, 2, 64, 16, seed=54)
    dw = DeviceWorkload(w)
    t = w.table.copy()
    t.indices[1] = w.table.num_total_pages + 5
    dw.set_table(t)
    dw.decode()
    torch.cuda.synchronize()
    assert dw.flags() & pd.PD_FLAG_BAD_PAGE_ID
    pd.pd_workspace_init(dw.ws)
    t2 = w.table.copy()
    t2.last_page_len[0] = 99
    dw.set_table(t2)
    dw.decode()
    assert dw.flags() == pd.PD_FLAG_BAD_LAST_PAGE_LEN
    pd.pd_workspace_init(dw.ws)
    t3 = w.table.copy()
    t3.indptr[2] = t3.indptr[1] - 1
    dw.set_table(t3)
    dw.decode()
    assert dw.flags() & pd.PD_FLAG_BAD_INDPTR


@pytest.mark.parametrize("how", ["a range ends before it starts", "indptr[batch] below indptr[0]"])
def test_decreasing_indptr_is_flagged_and_the_next_call_is_clean(how):
    """A decreasing indptr on the tensor-core kernel (group 4, pages of 16
    rows), whose first copies go out before the table is staged, with shares
    long enough to take tails. The call finishes and sets PD_FLAG_BAD_INDPTR
    (its outputs are then undefined); the next call with the good table, on the
    same workspace after pd_workspace_init, gives bit for bit what it gave
    before the bad call, with no flag: the context, the workspace and its tail
    counters are intact."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.llama3_8b_bf16(seed=57, batch=24, lo=1000, hi=4000)
    dw = DeviceWorkload(w)
    o_good, l_good = (x.clone() for x in dw.decode())
    compare(o_good, l_good, *oracle.paged_decode_workload(w), "bf16", "good table")
    bad = w.table.copy()
    if how == "a range ends before it starts":
        bad.indptr[5] = bad.indptr[4] - 50
    else:
        bad.indptr[0] = 40
        bad.indptr[-1] = 20
    dw.set_table(bad)
    dw.decode()
    assert dw.flags() & pd.PD_FLAG_BAD_INDPTR
    pd.pd_workspace_init(dw.ws)
    dw.set_table(w.table)
    o2, l2 = dw.decode()
    assert dw.flags() == 0
    assert torch.equal(o2.view(torch.int16), o_good.view(torch.int16)) and torch.equal(l2, l_good)


def test_repeated_calls_are_bit_identical():
    import torch

    w = wl.llama3_8b_bf16(seed=55, batch=8, lo=100, hi=3000)
    dw = DeviceWorkload(w)
    o1, l1 = (x.clone() for x in dw.decode())
    for _ in range(3):
        o2, l2 = dw.decode()
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1, l2)


def test_result_ignores_nan_in_unused_rows():
    # Poisoned rows (past last_page_len, unused pages) are NaN; output stays finite
    # and equals the result with those rows set to random finite values.
    import torch

    w = wl.make_paged("poison", "bf16", [17, 33, 48, 5], 16, 4, 128, 16, seed=56)
    dw = DeviceWorkload(w)
    o1 = dw.decode()[0].clone()
    k2 = np.where(w.k_data == np.uint16(0x7FC0), np.uint16(0x3F80), w.k_data)
    v2 = np.where(w.v_data == np.uint16(0x7FC0), np.uint16(0xC000), w.v_data)
    dw.k = to_dev(k2, "bf16")
    dw.v = to_dev(v2, "bf16")
    o2 = dw.decode()[0]
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


# --- contiguous entry ----------------------------------------------------------------------

@pytest.mark.parametrize("dtype,valid,maxlen", [("f16", 5000, 5000), ("bf16", 777, 1000), ("f32", 64, 64),
                                                 ("f16", 1, 33)])
def test_contiguous_decode_matches_oracle(dtype, valid, maxlen):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    B, Hq, Hk, D = 3, 32, 8, 128
    key = wl.stream_key(60 + valid, "k")
    kc = wl.normal((B, Hk, maxlen, D), dtype, key)
    vc = wl.normal((B, Hk, maxlen, D), dtype, wl.stream_key(60 + valid, "v"))
    q = wl.normal((B, Hq, D), dtype, wl.stream_key(60 + valid, "q"))
    nan = wl.nan_value(dtype)
    kc[:, :, valid:] = nan
    vc[:, :, valid:] = nan
    scale = float(np.float32(1 / math.sqrt(D)))
    o_ref, lse_ref = oracle.contiguous_decode(q, kc, vc, Hq, valid, scale, dtype)
    qd, kd, vd = to_dev(q, dtype), to_dev(kc, dtype), to_dev(vc, dtype)
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(B, Hq, Hk, D, code))
    pd.pd_contiguous_decode(qd, kd, vd, o, lse, valid, scale, ws)
    compare(o, lse, o_ref, lse_ref, dtype, "contiguous")
    o2 = torch.empty_like(qd)
    pd.pd_contiguous_decode(qd, kd, vd, o2, None, valid, scale, ws)  # lse is optional
    assert torch.equal(o.view(torch.int16) if dtype != "f32" else o, o2.view(torch.int16) if dtype != "f32" else o2)


def test_contiguous_zero_valid_rows():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    q = torch.randn(2, 8, 64, device="cuda", dtype=torch.float16)
    k = torch.randn(2, 2, 10, 64, device="cuda", dtype=torch.float16)
    o = torch.full_like(q, 7.0)
    lse = torch.zeros(2, 8, device="cuda")
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(2, 8, 2, 64, pd.PD_F16))
    pd.pd_contiguous_decode(q, k, k, o, lse, 0, 0.125, ws)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_contiguous_equals_paged_on_the_same_values():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.long_context_f16(seed=61, batch=2, kv_len=3000)
    kc, vc, n = wl.contiguous_copy(w)
    dw = DeviceWorkload(w)
    o1, l1 = dw.decode()
    o2 = torch.empty_like(dw.q)
    l2 = torch.empty_like(dw.lse)
    ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(w.batch, 32, 8, 128, pd.PD_F16))
    pd.pd_contiguous_decode(dw.q, to_dev(kc, "f16"), to_dev(vc, "f16"), o2, l2, n, w.sm_scale, ws)
    o_ref, lse_ref = oracle.paged_decode_workload(w)
    compare(o2, l2, o_ref, lse_ref, "f16", "contiguous vs oracle")
    assert float((o1.float() - o2.float()).abs().max()) <= 2 * O_TOL["f16"]


# --- merge of partial states ---------------------------------------------------------------

@pytest.mark.parametrize("dtype,head_dim,parts", [("bf16", 128, 2), ("f16", 256, 7), ("f32", 64, 40)])
def test_merge_states_matches_oracle_merge(dtype, head_dim, parts):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    # Oracle partial states over disjoint token sets (page_size 1: one token per page).
    rng = np.random.default_rng(70 + parts)
    Hq, Hk, n = 8, 2, 300
    k = wl.normal((n, Hk, 1, head_dim), dtype, wl.stream_key(70, "k"))
    v = wl.normal((n, Hk, 1, head_dim), dtype, wl.stream_key(70, "v"))
    q1 = wl.normal((1, Hq, head_dim), dtype, wl.stream_key(70, "q"))
    owner = rng.integers(0, parts, n)
    sets = [np.flatnonzero(owner == c) for c in range(parts)]
    indices = np.concatenate(sets).astype(np.int32)
    indptr = np.cumsum([0] + [len(s) for s in sets]).astype(np.int32)
    lpl = np.ones(parts, dtype=np.int32)
    scale = float(np.float32(1 / math.sqrt(head_dim)))
    op, lp = oracle.paged_decode(np.repeat(q1, parts, 0), k, v, indices, indptr, lpl, Hq, Hk, head_dim, 1,
                                 scale, dtype)
    op32 = op.astype(np.float32)
    lp32 = lp.astype(np.float32)
    om, lm = oracle.merge_states(op32.astype(np.float64), lp32.astype(np.float64))
    o = torch.empty(Hq, head_dim, dtype={"f32": torch.float32, "f16": torch.float16,
                                          "bf16": torch.bfloat16}[dtype], device="cuda")
    lse = torch.empty(Hq, device="cuda")
    pd.pd_merge_states(torch.from_numpy(op32).cuda(), torch.from_numpy(lp32).cuda(), o, lse)
    compare(o, lse, om, lm, dtype, "merge")
    # and the merge of the parts equals attention over all tokens
    of, lf = oracle.paged_decode(q1, k, v, np.arange(n, dtype=np.int32), np.array([0, n], np.int32),
                                 np.ones(1, np.int32), Hq, Hk, head_dim, 1, scale, dtype)
    compare(o, lse, of[0], lf[0], dtype, "merge vs full")


def test_merge_states_all_parts_empty():
    import torch

    import paged_kv_gqa_13_gb300 as pd

    op = torch.zeros(3, 5, 128, device="cuda")
    lp = torch.full((3, 5), -math.inf, device="cuda")
    o = torch.full((5, 128), 3.0, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(5, device="cuda")
    pd.pd_merge_states(op, lp, o, lse)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("lead,trail", [(0, 5), (2, 1)])  # both hit on 148- and 152-SM grids
def test_indices_entries_that_no_request_lists(lead, trail):
    """`indices` may hold entries outside [indptr[0], indptr[batch]) (the header
    allows indptr[batch] < num_indices). Those positions have no chunk; with ~5
    positions per warp, some warps start among them and run into the next
    pass's listed pages, which the early first copies must not mistake for
    their first chunks."""
    import dataclasses

    w = wl.make_paged("unlisted", "bf16", [2400, 2390, 2401, 2397], 32, 8, 128, 16, seed=96)
    t = w.table
    filler = t.indices[:max(lead, trail)]  # valid page ids that no request lists here
    t2 = dataclasses.replace(t, indices=np.concatenate([filler[:lead], t.indices, filler[:trail]]).astype(np.int32),
                             indptr=(t.indptr + lead).astype(np.int32))
    dw = DeviceWorkload(w)
    dw.set_table(t2)
    o, lse = dw.decode()
    assert dw.flags() == 0
    o_ref, lse_ref = oracle.paged_decode(w.q, w.k_data, w.v_data, t2.indices, t2.indptr, t2.last_page_len,
                                         w.num_qo_heads, w.num_kv_heads, w.head_dim, t2.page_size, w.sm_scale, "bf16")
    compare(o, lse, o_ref, lse_ref, "bf16", f"{lead} leading, {trail} trailing unlisted entries")
