"""Pins for the CPU oracle: each test checks it against a fact the problem or
the mathematics fixes, never against the oracle itself.

What each pin would catch is noted beside it (a dropped term, a wrong sign or
index, a transposed operand).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NINF = -math.inf


def _table(kv_len, P, pool, seed=0):
    return wl.build_page_table(np.asarray(kv_len), P, pool, np.random.default_rng(seed))


def _rand(shape, dtype, seed, stream="k"):
    return wl.normal(shape, dtype, wl.stream_key(seed, stream))


def _decode(w_q, k, v, t, Hq, Hk, D, scale, dtype, threads=0):
    return oracle.paged_decode(w_q, k, v, t.indices, t.indptr, t.last_page_len, Hq, Hk, D,
                               t.page_size, scale, dtype, threads)


def _vals(raw, dtype):
    return oracle.decode_elements(raw, dtype)


# --- element decoding: reduces to a library routine ------------------------------------------

def test_decode_f16_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_elements(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))  # catches a lost sign


def test_decode_bf16_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32)
    got = oracle.decode_elements(bits.astype(np.uint16), "bf16")
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_decode_f32_roundtrip():
    x = np.random.default_rng(1).standard_normal(4096).astype(np.float32) * 1e3
    assert np.array_equal(oracle.decode_elements(x, "f32"), x.astype(np.float64))


def _nearest_even(x, table_vals, table_bits):
    """Brute force: nearest representable value, ties to the even bit pattern."""
    order = np.argsort(table_vals)
    tv, tb = table_vals[order], table_bits[order]
    out = []
    for v in x:
        i = np.searchsorted(tv, v)
        cands = [j for j in (i - 1, i) if 0 <= j < len(tv)]
        best = min(cands, key=lambda j: (abs(tv[j] - v), int(tb[j]) & 1))
        out.append(tb[best])
    return np.asarray(out, dtype=np.uint16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_round_to_dtype_is_nearest_even(dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode_elements(bits, dtype)
    keep = np.isfinite(vals) & ~((vals == 0) & np.signbit(vals))
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(3000) * 4, rng.standard_normal(500) * 1e-6,
                        (vals[keep][rng.integers(0, keep.sum(), 500)] +
                         vals[keep][rng.integers(0, keep.sum(), 500)]) / 2])
    x = x[np.abs(x) < 60000]
    got = oracle.round_to_dtype(x, dtype)
    want = _nearest_even(x, vals[keep], bits[keep])
    assert np.array_equal(oracle.decode_elements(got, dtype), oracle.decode_elements(want, dtype))
    if dtype == "f16":
        assert np.array_equal(got, x.astype(np.float16).view(np.uint16))


# --- closed forms --------------------------------------------------------------------------

def _onehot_q(B, Hq, D, dtype, coef=2.0):
    """q[b, h] = coef at dimension h % D, zero elsewhere: the score is coef * k[h % D]."""
    q = np.zeros((B, Hq, D), dtype=np.float32)
    for h in range(Hq):
        q[:, h, h % D] = coef
    return wl.round_f32(q, dtype)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_kv_len_one_returns_its_v_row_and_lse_is_its_score(dtype):
    # Catches: a wrong V row or head, a missing sm_scale, lse in log2 instead of ln.
    B, Hq, Hk, D, P = 3, 8, 2, 64, 16
    t = _table([1, 1, 1], P, 12, seed=3)
    k = _rand((12, Hk, P, D), dtype, 4, "k")
    v = _rand((12, Hk, P, D), dtype, 4, "v")
    q = _onehot_q(B, Hq, D, dtype)
    scale = 0.125
    o, lse = _decode(q, k, v, t, Hq, Hk, D, scale, dtype)
    kv, vv = _vals(k, dtype), _vals(v, dtype)
    for b in range(B):
        page = t.indices[t.indptr[b]]
        for h in range(Hq):
            kh = h // (Hq // Hk)
            assert np.array_equal(o[b, h], vv[page, kh, 0])
            assert lse[b, h] == scale * 2.0 * kv[page, kh, 0, h % D]


def test_identical_k_rows_give_mean_of_v_and_lse_plus_ln_n():
    # Catches: a dropped normalisation, a wrong count of rows, an off-by-one in the walk.
    Hq, Hk, D, P = 4, 2, 64, 16
    n = 37
    t = _table([n], P, 8, seed=5)
    k = _rand((8, Hk, P, D), "bf16", 6, "k")
    row = _rand((Hk, D), "bf16", 7, "k")
    for p in t.indices:
        k[p] = row[:, None, :]
    v = _rand((8, Hk, P, D), "bf16", 6, "v")
    q = _onehot_q(1, Hq, D, "bf16", coef=3.0)
    o, lse = _decode(q, k, v, t, Hq, Hk, D, 0.125, "bf16")
    vv, rv = _vals(v, "bf16"), _vals(row, "bf16")
    for h in range(Hq):
        kh = h // 2
        rows = [vv[t.indices[i // P], kh, i % P] for i in range(n)]
        np.testing.assert_allclose(o[0, h], np.mean(rows, axis=0), rtol=0, atol=1e-14)
        s = 0.125 * 3.0 * rv[kh, h % D]
        assert abs(lse[0, h] - (s + math.log(n))) < 1e-13


def test_gqa_decode_constant_example_closed_form():
    # The one input the pages print (ferrox-cuda attn.rs test): constant q, k, v.
    ex = json.load(open(os.path.join(GOLDEN, "gqa_decode_constant_example.json")))["inputs"]
    H, Hk, D, n = ex["n_heads"], ex["n_kv_heads"], ex["head_dim"], ex["seq_len"]
    qv, kv, vv = (np.float32(ex[x]) for x in ("q", "k", "v"))
    scale = np.float32(1.0 / math.sqrt(D))
    P = 4
    t = _table([n], P, 1, seed=0)
    q = np.full((1, H, D), qv, dtype=np.float32)
    k = np.full((1, Hk, P, D), kv, dtype=np.float32)
    v = np.full((1, Hk, P, D), vv, dtype=np.float32)
    o, lse = _decode(q, k, v, t, H, Hk, D, scale, "f32")
    assert np.all(o == np.float64(vv))
    s = float(scale) * D * float(qv) * float(kv)
    np.testing.assert_allclose(lse, s + math.log(n), rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - (5.6568542e-4 + math.log(3))) < 1e-9  # the value worked out by hand


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_log_sum_exp_and_output(seed):
    # Brute force on tiny inputs: no max shift, exact summation (math.fsum), plain loops.
    # Catches: a wrong max, a dropped term, exp of unscaled scores, a transposed V.
    rng = np.random.default_rng(10 + seed)
    Hq, Hk, D, P = 2, 1, 8, 4
    lens = [int(rng.integers(1, 40)), int(rng.integers(1, 40))]
    t = _table(lens, P, 24, seed=seed)
    q = (rng.standard_normal((2, Hq, D)) * 0.8).astype(np.float32)
    k = (rng.standard_normal((24, Hk, P, D)) * 0.8).astype(np.float32)
    v = rng.standard_normal((24, Hk, P, D)).astype(np.float32)
    scale = np.float32(0.35)
    o, lse = _decode(q, k, v, t, Hq, Hk, D, scale, "f32")
    for b in range(2):
        rows = [(t.indices[t.indptr[b] + i // P], i % P) for i in range(lens[b])]
        for h in range(Hq):
            s = [float(scale) * math.fsum(float(q[b, h, d]) * float(k[p, 0, r, d]) for d in range(D))
                 for p, r in rows]
            e = [math.exp(x) for x in s]
            Z = math.fsum(e)
            assert abs(lse[b, h] - math.log(Z)) < 1e-12
            for d in range(D):
                want = math.fsum(e[i] * float(v[p, 0, r, d]) for i, (p, r) in enumerate(rows)) / Z
                assert abs(o[b, h, d] - want) < 1e-12


# --- invariants ----------------------------------------------------------------------------

def test_invariant_under_permutation_of_physical_page_ids():
    # Catches: reading page p instead of indices[i], or any dependence on physical order.
    w = wl.llama3_8b_bf16(seed=21, batch=3, lo=20, hi=90)
    o1, l1 = oracle.paged_decode_workload(w)
    pi = np.random.default_rng(22).permutation(w.table.num_total_pages).astype(np.int32)
    k2 = np.empty_like(w.k_data)
    v2 = np.empty_like(w.v_data)
    k2[pi] = w.k_data
    v2[pi] = w.v_data
    t = w.table
    o2, l2 = oracle.paged_decode(w.q, k2, v2, pi[t.indices], t.indptr, t.last_page_len,
                                 w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size,
                                 w.sm_scale, w.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_equals_contiguous_path():
    # Two code paths (page walk vs direct rows). Catches: row t % P / page t // P swapped.
    w = wl.long_context_f16(seed=23, batch=2, kv_len=77)
    kc, vc, n = wl.contiguous_copy(w, max_kv_len=96)
    o1, l1 = oracle.paged_decode_workload(w)
    o2, l2 = oracle.contiguous_decode(w.q, kc, vc, w.num_qo_heads, n, w.sm_scale, w.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gqa_equals_mha_with_replicated_kv_heads():
    # Catches: kv head h % Hk instead of h // group.
    w = wl.ragged_70b_bf16(seed=24, batch=4, max_len=100)
    g = w.group
    t = w.table
    k2 = np.repeat(w.k_data, g, axis=1)
    v2 = np.repeat(w.v_data, g, axis=1)
    o1, l1 = oracle.paged_decode_workload(w)
    o2, l2 = oracle.paged_decode(w.q, k2, v2, t.indices, t.indptr, t.last_page_len,
                                 w.num_qo_heads, w.num_qo_heads, w.head_dim, t.page_size,
                                 w.sm_scale, w.dtype)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_output_is_linear_in_v():
    # Catches: V weights not normalised by the same Z as lse, or a V term dropped.
    rng = np.random.default_rng(25)
    Hq, Hk, D, P = 4, 2, 64, 16
    t = _table([50, 3], P, 8, seed=25)
    q = rng.standard_normal((2, Hq, D)).astype(np.float32)
    k = rng.standard_normal((8, Hk, P, D)).astype(np.float32)
    v1 = (rng.integers(-64, 64, (8, Hk, P, D)) / 8.0).astype(np.float32)
    v2 = (rng.integers(-64, 64, (8, Hk, P, D)) / 8.0).astype(np.float32)
    a, _ = _decode(q, k, v1, t, Hq, Hk, D, 0.125, "f32")
    b, _ = _decode(q, k, v2, t, Hq, Hk, D, 0.125, "f32")
    c, _ = _decode(q, k, (3 * v1 - 2 * v2).astype(np.float32), t, Hq, Hk, D, 0.125, "f32")
    np.testing.assert_allclose(c, 3 * a - 2 * b, rtol=0, atol=1e-12)


def test_one_dominant_key_selects_its_value_row():
    # A key aligned with q scores > 50 above the rest: o is that key's V row.
    # Catches: P.V using the wrong token index (e.g. page order instead of list order).
    rng = np.random.default_rng(26)
    Hq, Hk, D, P = 2, 1, 64, 16
    n = 45
    t = _table([n], P, 5, seed=26)
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    q[0, 1] = q[0, 0]
    k = (rng.standard_normal((5, Hk, P, D)) * 0.1).astype(np.float32)
    v = rng.standard_normal((5, Hk, P, D)).astype(np.float32)
    j = 29
    pj, rj = t.indices[j // P], j % P
    k[pj, 0, rj] = q[0, 0] * (80.0 / float(np.dot(q[0, 0], q[0, 0]) * 0.125))
    o, lse = _decode(q, k, v, t, Hq, Hk, D, 0.125, "f32")
    np.testing.assert_allclose(o[0, 0], v[pj, 0, rj].astype(np.float64), rtol=0, atol=1e-15)


def test_merge_of_disjoint_token_sets_equals_full():
    # page_size 1 makes every token its own page, so the split is at token level.
    # Catches: a wrong sign in exp(lse_c - L), a missing log, merging in log2.
    rng = np.random.default_rng(27)
    Hq, Hk, D, P = 4, 2, 64, 1
    n = 60
    k = rng.standard_normal((n, Hk, P, D)).astype(np.float32)
    v = rng.standard_normal((n, Hk, P, D)).astype(np.float32)
    q1 = rng.standard_normal((1, Hq, D)).astype(np.float32)
    mask = rng.random(n) < 0.4
    sets = [np.arange(n), np.flatnonzero(mask), np.flatnonzero(~mask)]
    indices = np.concatenate(sets).astype(np.int32)
    indptr = np.cumsum([0] + [len(s) for s in sets]).astype(np.int32)
    lpl = np.ones(3, dtype=np.int32)
    q = np.repeat(q1, 3, axis=0)
    o, lse = oracle.paged_decode(q, k, v, indices, indptr, lpl, Hq, Hk, D, P, 0.125, "f32")
    om, lm = oracle.merge_states(o[1:], lse[1:])
    np.testing.assert_allclose(om, o[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lse[0], rtol=0, atol=1e-13)
    # Merging with an empty part changes nothing.
    oe, le = oracle.merge_states(np.stack([o[0], np.zeros_like(o[0])]), np.stack([lse[0], np.full(Hq, NINF)]))
    np.testing.assert_allclose(oe, o[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(le, lse[0], rtol=0, atol=1e-15)
    oz, lz = oracle.merge_states(np.zeros((2, Hq, D)), np.full((2, Hq), NINF))
    assert np.all(oz == 0) and np.all(lz == NINF)


# --- special cases of the page table -------------------------------------------------------

def test_empty_requests_give_zero_and_minus_inf():
    Hq, Hk, D, P = 4, 2, 64, 16
    k = _rand((6, Hk, P, D), "f16", 30, "k")
    v = _rand((6, Hk, P, D), "f16", 30, "v")
    q = _rand((3, Hq, D), "f16", 30, "q")
    indices = np.array([4, 2], dtype=np.int32)
    indptr = np.array([0, 0, 1, 2], dtype=np.int32)  # b0: no pages, b1: one page with 0 rows
    lpl = np.array([0, 0, 5], dtype=np.int32)
    o, lse = oracle.paged_decode(q, k, v, indices, indptr, lpl, Hq, Hk, D, P, 0.125, "f16")
    assert np.all(o[:2] == 0) and np.all(lse[:2] == NINF)
    assert np.all(np.isfinite(lse[2]))


def test_last_page_len_zero_drops_the_last_page():
    Hq, Hk, D, P = 4, 2, 64, 16
    k = _rand((6, Hk, P, D), "bf16", 31, "k")
    v = _rand((6, Hk, P, D), "bf16", 31, "v")
    q = _rand((2, Hq, D), "bf16", 31, "q")
    indices = np.array([3, 1, 5, 3, 1], dtype=np.int32)
    indptr = np.array([0, 3, 5], dtype=np.int32)
    lpl = np.array([0, P], dtype=np.int32)  # b0: pages 3,1 full + empty page 5 == b1
    o, lse = oracle.paged_decode(q[[0, 0]], k, v, indices, indptr, lpl, Hq, Hk, D, P, 0.125, "bf16")
    assert np.array_equal(o[0], o[1]) and np.array_equal(lse[0], lse[1])


def test_rejects_bad_tables_and_descriptors():
    Hq, Hk, D, P = 4, 2, 64, 16
    k = np.zeros((4, Hk, P, D), dtype=np.float32)
    q = np.zeros((1, Hq, D), dtype=np.float32)
    ok = dict(indices=[0, 1], indptr=[0, 2], last_page_len=[3])
    oracle.paged_decode(q, k, k, num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D, page_size=P,
                        sm_scale=1.0, dtype="f32", **ok)
    for bad in (dict(indices=[0, 4]), dict(indices=[-1, 0]), dict(last_page_len=[17]),
                dict(indptr=[0, 3])):
        args = dict(ok, **bad)
        with pytest.raises(oracle.OracleError):
            oracle.paged_decode(q, k, k, num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D, page_size=P,
                                sm_scale=1.0, dtype="f32", **args)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, k, k, num_qo_heads=3, num_kv_heads=2, head_dim=D, page_size=P,
                            sm_scale=1.0, dtype="f32", **ok)


def test_result_does_not_depend_on_thread_count():
    w = wl.llama3_8b_bf16(seed=32, batch=4, lo=30, hi=200)
    a = oracle.paged_decode_workload(w, threads=1)
    b = oracle.paged_decode_workload(w, threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --- append --------------------------------------------------------------------------------

def test_append_writes_the_new_last_token():
    # After the caller's table update and the append, the new row is the last token:
    # a query aligned with the new key selects the new value row.
    # Catches: writing at last_page_len instead of last_page_len - 1, or into the old page.
    w = wl.mha_append_f16(seed=33, batch=5, lo=1, hi=40, steps=3)
    k, v = w.k_data.copy(), w.v_data.copy()
    t = w.table
    for step in range(3):
        t2 = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        before_k = k.copy()
        oracle.paged_append(kn, vn, k, v, t2.indices, t2.indptr, t2.last_page_len, w.dtype)
        changed = np.argwhere(np.any(k.view(np.uint16) != before_k.view(np.uint16), axis=-1))
        assert len(changed) <= w.batch * w.num_kv_heads  # only the new rows moved
        t = t2
        # q = new key * large factor makes the new token dominant for every head.
        knv = oracle.decode_elements(kn, "f16")
        qf = (knv * (60.0 / np.maximum((knv * knv).sum(-1, keepdims=True) * w.sm_scale, 1e-3)))
        q = wl.round_f32(qf.astype(np.float32), "f16")
        o, lse = oracle.paged_decode(q, k, v, t.indices, t.indptr, t.last_page_len, w.num_qo_heads,
                                     w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale, "f16")
        vnv = oracle.decode_elements(vn, "f16")
        np.testing.assert_allclose(o, vnv, rtol=0, atol=1e-6)


def test_contiguous_append_writes_the_new_last_row():
    # After appending at position n, a contiguous decode over n + 1 rows with a
    # query aligned to the new key returns the new value row, and only the new
    # rows of the cache changed. Catches: writing row n - 1 or row n + 1.
    B, Hk, L, D, n = 3, 4, 40, 64, 25
    kc = wl.normal((B, Hk, L, D), "f16", wl.stream_key(140, "k"))
    vc = wl.normal((B, Hk, L, D), "f16", wl.stream_key(140, "v"))
    kn = wl.normal((B, Hk, D), "f16", wl.stream_key(140, "k_new"))
    vn = wl.normal((B, Hk, D), "f16", wl.stream_key(140, "v_new"))
    before = kc.copy()
    oracle.contiguous_append(kn, vn, kc, vc, n, "f16")
    changed = np.argwhere(np.any(kc != before, axis=-1))
    assert {tuple(x[2:]) for x in changed} == {(n,)}
    knv = oracle.decode_elements(kn, "f16")
    qf = knv * (60.0 / np.maximum((knv * knv).sum(-1, keepdims=True) * 0.125, 1e-3))
    q = wl.round_f32(qf.astype(np.float32), "f16")
    o, _ = oracle.contiguous_decode(q, kc, vc, Hk, n + 1, 0.125, "f16")
    np.testing.assert_allclose(o, oracle.decode_elements(vn, "f16"), rtol=0, atol=1e-6)
    with pytest.raises(oracle.OracleError):
        oracle.contiguous_append(kn, vn, kc, vc, L, "f16")


def test_nhd_decode_reads_token_t_of_head_kh_at_the_page_offset():
    # ferrox-cuda, src/attn.rs (gqa_decode): token t of kv head kv_h starts at
    # element (t * n_kv_heads + kv_h) * head_dim. Plant one dominant key at
    # token t0 of kv head 1, aligned with the query, and give every row of V
    # its own flat offset as its value: the q heads of kv head 1 must return
    # the V row at that offset, the others the mean of their V rows.
    B, Hk, L, D, g, t0 = 2, 3, 7, 4, 2, 5
    Hq = Hk * g
    flat_k = np.zeros(B * L * Hk * D, dtype=np.float32)
    flat_v = np.arange(B * L * Hk * D, dtype=np.float32) / D  # row r holds r, r + 1/D, ...
    q = np.zeros((B, Hq, D), dtype=np.float32)
    for b in range(B):
        off = ((b * L + t0) * Hk + 1) * D
        flat_k[off:off + D] = 8.0
        q[b, 1 * g:2 * g, :] = 8.0
    kc = flat_k.reshape(B, L, Hk, D)
    vc = flat_v.reshape(B, L, Hk, D)
    o, lse = oracle.contiguous_decode(q, kc, vc, Hq, L, 1.0, "f32", layout="nhd")
    for b in range(B):
        row = (b * L + t0) * Hk + 1
        np.testing.assert_allclose(o[b, g:2 * g], np.tile(flat_v[row * D:(row + 1) * D], (g, 1)), atol=1e-9)
        for kh in (0, 2):  # all scores 0: the plain mean of the kv head's rows
            rows = [(b * L + t) * Hk + kh for t in range(L)]
            mean = np.mean([flat_v[r * D:(r + 1) * D] for r in rows], axis=0)
            np.testing.assert_allclose(o[b, kh * g], mean, atol=1e-12)
            assert abs(lse[b, kh * g] - math.log(L)) < 1e-12


def test_nhd_decode_equals_hnd_decode_of_the_transposed_cache():
    # The layout changes only where a (token, head) row lives, never its value.
    B, Hq, Hk, L, D, n = 2, 8, 2, 50, 64, 37
    kc = wl.normal((B, L, Hk, D), "bf16", wl.stream_key(141, "k"))
    vc = wl.normal((B, L, Hk, D), "bf16", wl.stream_key(141, "v"))
    q = wl.normal((B, Hq, D), "bf16", wl.stream_key(141, "q"))
    o1, l1 = oracle.contiguous_decode(q, kc, vc, Hq, n, 0.125, "bf16", layout="nhd")
    o2, l2 = oracle.contiguous_decode(q, np.ascontiguousarray(kc.transpose(0, 2, 1, 3)),
                                      np.ascontiguousarray(vc.transpose(0, 2, 1, 3)), Hq, n, 0.125, "bf16")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_nhd_append_writes_token_position_of_every_head():
    B, Hk, L, D, n = 2, 3, 9, 8, 6
    kc = wl.normal((B, L, Hk, D), "f16", wl.stream_key(142, "k"))
    vc = wl.normal((B, L, Hk, D), "f16", wl.stream_key(142, "v"))
    kn = wl.normal((B, Hk, D), "f16", wl.stream_key(142, "k_new"))
    vn = wl.normal((B, Hk, D), "f16", wl.stream_key(142, "v_new"))
    kb, vb = kc.copy(), vc.copy()
    oracle.contiguous_append(kn, vn, kc, vc, n, "f16", layout="nhd")
    fk, fkb = kc.reshape(-1), kb.reshape(-1)
    for b in range(B):
        for h in range(Hk):
            off = ((b * L + n) * Hk + h) * D  # the page's token-major offset
            assert np.array_equal(fk[off:off + D], kn[b, h])
            fkb[off:off + D] = kn[b, h]
    assert np.array_equal(fk, fkb)  # nothing else changed
    assert np.array_equal(vc[:, n], vn) and np.array_equal(np.delete(vc, n, axis=1), np.delete(vb, n, axis=1))


# --- FP8 E4M3 pools: value = code value * per-kv-head scale ---------------------------------
# The code values follow the OCP 8-bit floating point specification (OFP8), E4M3:
# bias 7, 3 mantissa bits, subnormals (m/8)*2^-6, S.1111.111 NaN, no infinity.

def test_e4m3_values_at_the_format_anchors():
    anchors = {0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x0F: 1.875 * 2.0**-6,
               0x30: 0.5, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0}
    codes = np.array(list(anchors), dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_values(codes), np.array(list(anchors.values())))
    assert np.array_equal(oracle.e4m3_values(codes | 0x80), -np.array(list(anchors.values())))
    allv = oracle.e4m3_values(np.arange(256, dtype=np.uint8))
    assert set(np.flatnonzero(np.isnan(allv))) == {0x7F, 0xFF}
    pos = allv[:0x7F]
    assert np.all(np.diff(pos) > 0)  # magnitudes increase with the code
    assert np.signbit(allv[0x80]) and allv[0x80] == 0.0
    fin = allv[~np.isnan(allv)]
    assert np.array_equal(fin.astype(np.float16).astype(np.float64), fin)  # every value is an f16


def test_e4m3_round_is_nearest_even_and_saturates():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle.e4m3_values(codes)
    assert np.array_equal(oracle.e4m3_round(vals.astype(np.float32)), codes)
    assert np.array_equal(oracle.e4m3_round(-vals[1:].astype(np.float32)), codes[1:] | 0x80)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact: one more mantissa bit
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[:-1] + 1)
    assert np.array_equal(oracle.e4m3_round(mids), even)
    assert np.array_equal(oracle.e4m3_round(np.nextafter(mids, np.float32(np.inf))), codes[1:])
    assert np.array_equal(oracle.e4m3_round(np.nextafter(mids, np.float32(0))), codes[:-1])
    big = np.array([448.0, 449.0, 464.0, 1e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert list(oracle.e4m3_round(big)) == [0x7E] * 5 + [0xFE] * 2
    assert oracle.e4m3_round(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def _fp8_workload(seed, q_dtype="f16", pow2_scales=False, lens=(0, 1, 15, 16, 17, 200), Hq=8, Hk=2, D=64, P=16):
    w = wl.make_paged(f"fp8_{seed}", q_dtype, list(lens), Hq, Hk, D, P, seed)
    k8, v8, ks, vs = wl.fp8_pool(w)
    if pow2_scales:
        ks = np.array([2.0 ** -(2 + h % 3) for h in range(Hk)], dtype=np.float32)
        vs = np.array([2.0 ** -(1 + h % 4) for h in range(Hk)], dtype=np.float32)
    return w, k8, v8, ks, vs


def _fp8_decode(w, k8, v8, ks, vs, q=None, sm_scale=None):
    t = w.table
    return oracle.paged_decode_fp8(w.q if q is None else q, k8, v8, ks, vs, t.indices, t.indptr, t.last_page_len,
                                   w.num_qo_heads, w.num_kv_heads, w.head_dim, t.page_size,
                                   w.sm_scale if sm_scale is None else sm_scale, w.dtype)


def test_fp8_decode_equals_f32_decode_of_the_dequantised_pool():
    # With power-of-two scales every code value * scale is exact in f32, so the
    # FP8 decode must equal, bit for bit, the f32 decode (pinned above) over a
    # pool holding those values. NaN codes in unused rows become NaN values there.
    w, k8, v8, ks, vs = _fp8_workload(150, pow2_scales=True)
    o8, l8 = _fp8_decode(w, k8, v8, ks, vs)
    h = np.arange(w.num_kv_heads)[None, :, None, None]
    k32 = (oracle.e4m3_values(k8) * ks[h]).astype(np.float32)
    v32 = (oracle.e4m3_values(v8) * vs[h]).astype(np.float32)
    q32 = oracle.decode_elements(w.q, "f16").astype(np.float32)
    t = w.table
    o32, l32 = oracle.paged_decode(q32, k32, v32, t.indices, t.indptr, t.last_page_len, w.num_qo_heads,
                                   w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale, "f32")
    assert np.array_equal(o8, o32) and np.array_equal(l8, l32)


def test_fp8_scales_act_per_kv_head():
    # v_scale[h] scales the outputs of kv head h's q heads and nothing else;
    # k_scale[h] acts like sm_scale for those heads.
    w, k8, v8, ks, vs = _fp8_workload(151, q_dtype="bf16")
    g = w.num_qo_heads // w.num_kv_heads
    o, l = _fp8_decode(w, k8, v8, ks, vs)
    vs2 = vs.copy()
    vs2[1] *= 2
    o2, l2 = _fp8_decode(w, k8, v8, ks, vs2)
    np.testing.assert_allclose(o2[:, g:2 * g], 2 * o[:, g:2 * g], rtol=1e-14, atol=0)
    assert np.array_equal(o2[:, :g], o[:, :g]) and np.array_equal(l2, l)
    ks3 = np.full_like(ks, ks[0])
    o3, l3 = _fp8_decode(w, k8, v8, ks3, vs, sm_scale=np.float32(w.sm_scale * 2))
    ks4 = np.full_like(ks, 2 * ks[0])
    o4, l4 = _fp8_decode(w, k8, v8, ks4, vs)
    np.testing.assert_allclose(o3, o4, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l3, l4, rtol=1e-12, atol=1e-14)


def test_fp8_append_rounds_the_f32_quotient():
    w, k8, v8, ks, vs = _fp8_workload(152, lens=(3, 16, 40))
    t = wl.table_after_append(w.table)
    kn, vn = w.new_rows(0)
    kb, vb = k8.copy(), v8.copy()
    oracle.paged_append_fp8(kn, vn, ks, vs, k8, v8, t.indices, t.indptr, t.last_page_len, "f16")
    kx = oracle.decode_elements(kn, "f16").astype(np.float32)
    changed = 0
    for b in range(w.batch):
        page = t.indices[t.indptr[b + 1] - 1]
        slot = t.last_page_len[b] - 1
        for h in range(w.num_kv_heads):
            quot = kx[b, h] / ks[h]  # f32 division
            got = k8[page, h, slot]
            err = np.abs(oracle.e4m3_values(got) - quot.astype(np.float64))
            # no other code is nearer to the quotient
            allv = oracle.e4m3_values(np.arange(256, dtype=np.uint8))
            best = np.nanmin(np.abs(allv[None, :] - quot.astype(np.float64)[:, None]), axis=1)
            assert np.all(err <= best)
            kb[page, h, slot] = got
            changed += 1
    assert np.array_equal(k8, kb)  # nothing but the new slots changed
    assert changed == w.batch * w.num_kv_heads
    assert not np.array_equal(v8, vb)
