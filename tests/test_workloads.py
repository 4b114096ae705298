"""The seeded input generator: determinism, rounding, page tables, poisoning."""
import numpy as np
import pytest

import workloads as wl


def test_splitmix64_reference_outputs():
    # splitmix64 with seed 0: the published first outputs of the generator.
    assert wl.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert wl.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert wl.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_normal_draws_are_thread_count_independent_and_sliceable():
    key = wl.stream_key(7, "k")
    a = wl.normal((300000,), "f32", key, threads=1)
    b = wl.normal((300000,), "f32", key, threads=8)
    assert np.array_equal(a, b)
    c = wl.normal((1000,), "f32", key, first=12345)
    assert np.array_equal(c, a[12345:13345])
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_storage_rounding_is_rne(dtype):
    x = np.random.default_rng(3).standard_normal(200000).astype(np.float32) * 3
    got = wl.round_f32(x, dtype)
    if dtype == "f16":
        assert np.array_equal(got, x.astype(np.float16).view(np.uint16))
    else:
        # Exhaustive neighbour check: the chosen bf16 is the nearest, ties to even.
        u = x.view(np.uint32)
        lo = (u >> 16).astype(np.uint32)
        hi = lo + 1
        vlo = (lo << 16).view(np.float32).astype(np.float64)
        vhi = (hi << 16).view(np.float32).astype(np.float64)
        xv = x.astype(np.float64)
        dlo, dhi = np.abs(xv - vlo), np.abs(xv - vhi)
        want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
        assert np.array_equal(got.astype(np.uint32), want)


def test_page_table_shape_and_shuffle():
    t = wl.build_page_table([100, 16, 1, 33], 16, 20, np.random.default_rng(0))
    assert list(t.indptr) == [0, 7, 8, 9, 12]
    assert list(t.last_page_len) == [4, 16, 1, 1]
    assert list(t.kv_len()) == [100, 16, 1, 33]
    assert len(set(t.indices.tolist())) == 12 and t.indices.max() < 20
    assert len(t.free_pages) == 8 and not set(t.free_pages) & set(t.indices.tolist())


def test_table_after_append_opens_a_page_only_when_full():
    t = wl.build_page_table([16, 5, 0], 16, 10, np.random.default_rng(1))
    t2 = wl.table_after_append(t)
    assert list(t2.kv_len()) == [17, 6, 1]
    assert list(t2.last_page_len) == [1, 6, 1]
    assert t2.indptr[1] - t2.indptr[0] == 2 and t2.indptr[3] - t2.indptr[2] == 1
    assert t2.indices[t2.indptr[1] - 1] == t.free_pages[0]
    assert np.array_equal(t2.indices[: t2.indptr[1] - 1], t.indices[: t.indptr[1]])


def test_workload_poisons_unused_rows_and_is_reproducible():
    a = wl.llama3_8b_bf16(seed=5, batch=3, lo=20, hi=70)
    b = wl.llama3_8b_bf16(seed=5, batch=3, lo=20, hi=70)
    assert np.array_equal(a.k_data, b.k_data) and np.array_equal(a.table.indices, b.table.indices)
    t = a.table
    nan = np.uint16(0x7FC0)
    used = set(t.indices.tolist())
    for p in range(t.num_total_pages):
        if p not in used:
            assert np.all(a.k_data[p] == nan)
    for bi in range(t.batch):
        last = t.indices[t.indptr[bi + 1] - 1]
        lpl = t.last_page_len[bi]
        assert np.all(a.v_data[last, :, lpl:] == nan)
        assert not np.any(a.v_data[last, :, :lpl] == nan)


def test_config_shapes():
    w = wl.tiny_gqa_f32()
    assert w.table.num_total_pages == 16 and list(w.table.kv_len()) == [100]
    assert w.table.num_indices == 7 and w.table.last_page_len[0] == 4
    assert w.sm_scale == 0.125
    r = wl.ragged_70b_bf16(batch=16, max_len=32768)
    assert list(r.table.kv_len()[:4]) == [1, 32, 64, 32768]
