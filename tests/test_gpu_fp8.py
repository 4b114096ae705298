"""GPU parity for FP8 (E4M3) pools with per-kv-head scales: the decode against
the oracle's FP8 decode, the append bit-exact against the oracle's quantiser."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import Fp8Device, compare, table_dev, to_dev

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 100, 3000, 33]


@pytest.mark.parametrize("dtype,Hq,Hk,D,P", [
    ("bf16", 32, 8, 128, 16),   # Llama-shaped group 4
    ("f16", 32, 8, 128, 16),
    ("bf16", 64, 8, 128, 32),   # group 8 (CUDA cores for E4M3)
    ("f16", 16, 16, 256, 16),   # MHA, D 256
    ("bf16", 16, 8, 64, 16),    # group 2, D 64
    ("f16", 24, 2, 128, 8),     # group 12: two head tiles, page 8
    ("bf16", 32, 8, 256, 16),   # group 4, D 256 (tensor cores)
    ("f16", 16, 8, 128, 16),    # group 2 (CUDA cores)
    ("bf16", 32, 8, 128, 1),    # one-row pages: two one-row chunks per stage
    ("f16", 64, 8, 128, 100),   # pages of 100 rows: 16-row chunks and a 4-row remainder
    ("bf16", 32, 8, 64, 16),    # group 4 at D 64 (CUDA cores)
])
def test_fp8_decode_matches_oracle(dtype, Hq, Hk, D, P):
    w = wl.make_paged(f"fp8_{dtype}_{Hq}_{Hk}_{D}", dtype, LENS, Hq, Hk, D, P, seed=300 + Hq + D + P)
    dev = Fp8Device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), dtype, "fp8 decode")
    import paged_kv_gqa_13_gb300 as pd

    assert pd.pd_read_device_flags(dev.ws) == 0


@pytest.mark.parametrize("dtype,Hq,Hk,D", [("bf16", 32, 8, 128), ("f16", 16, 16, 256), ("f16", 8, 2, 64)])
def test_fp8_append_then_decode(dtype, Hq, Hk, D):
    import paged_kv_gqa_13_gb300 as pd

    steps = 4
    w = wl.make_paged(f"fp8a_{dtype}", dtype, [0, 15, 16, 31, 200], Hq, Hk, D, 16, seed=320 + Hq,
                      extra_rows=steps, append_steps=steps)
    dev = Fp8Device(w)
    t = w.table
    for step in range(steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        dev.set_table(t)
        pd.pd_paged_append_fp8(to_dev(kn, dtype), to_dev(vn, dtype), dev.ksd, dev.vsd, dev.k, dev.v, dev.ind,
                               dev.ptr, dev.lpl, dev.ws)
        oracle.paged_append_fp8(kn, vn, dev.ks, dev.vs, dev.k8, dev.v8, t.indices, t.indptr, t.last_page_len,
                                dtype)
        assert np.array_equal(dev.k.cpu().numpy(), dev.k8), f"K codes differ, step {step}"
        assert np.array_equal(dev.v.cpu().numpy(), dev.v8), f"V codes differ, step {step}"
        o, lse = dev.decode()
        compare(o, lse, *dev.oracle_decode(), dtype, f"fp8 step {step}")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_fp8_append_saturates_and_rounds_ties_to_even():
    """Chosen quotients: exact codes, midpoints between codes, and values past 448."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("fp8_sat", "f16", [5], 8, 2, 64, 16, seed=331, extra_rows=1)
    dev = Fp8Device(w)
    t = wl.table_after_append(w.table)
    dev.set_table(t)
    ks = np.array([1.0, 0.5], dtype=np.float32)
    dev.ks, dev.ksd = ks, torch.from_numpy(ks).cuda()
    x = np.zeros((1, 2, 64), dtype=np.float32)
    x[0, :, :8] = [1.0, 1.0625, 1.125, 17.0, 448.0, 464.0, 1000.0, -0.0009765625]  # tie, tie, tie, ..., saturate
    x[0, :, 8:16] = [2.0**-9, 3 * 2.0**-10, 240.0, 232.0, -232.0, 0.3, -7.0, 65504.0]
    kn = wl.round_f32(x, "f16")
    vn = kn.copy()
    pd.pd_paged_append_fp8(to_dev(kn, "f16"), to_dev(vn, "f16"), dev.ksd, dev.vsd, dev.k, dev.v, dev.ind,
                           dev.ptr, dev.lpl, dev.ws)
    oracle.paged_append_fp8(kn, vn, dev.ks, dev.vs, dev.k8, dev.v8, t.indices, t.indptr, t.last_page_len, "f16")
    assert np.array_equal(dev.k.cpu().numpy(), dev.k8) and np.array_equal(dev.v.cpu().numpy(), dev.v8)


def test_fp8_cuda_core_kernel_with_share_tails():
    """E4M3 pool at group 2 (the CUDA-core kernel) with ~15 positions per warp,
    so that share tails are handed out: repeated calls agree bit for bit, the
    tail counters (workspace header bytes 64..71) return to zero, and the result
    matches the oracle."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("fp8_tails_g2", "f16", [16000, 1, 9000, 17, 8000], 16, 8, 128, 16, seed=78)
    dev = Fp8Device(w)
    o1, l1 = [t.clone() for t in dev.decode()]
    assert pd.pd_read_device_flags(dev.ws) == 0
    for _ in range(3):
        o, lse = dev.decode()
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, l1)
    assert dev.ws[64:72].view(torch.int32).cpu().tolist() == [0, 0]
    compare(o1, l1, *dev.oracle_decode(), w.dtype, "fp8 CUDA-core decode with share tails")


@pytest.mark.parametrize("dtype,Hq,Hk", [("bf16", 32, 8), ("f16", 16, 8)])
def test_fp8_batch_above_staged_table(dtype, Hq, Hk):
    """600 requests: indptr and last_page_len are read from global memory, not
    staged in shared memory; group 4 runs the E4M3 tensor-core kernel, group 2
    the CUDA-core variant."""
    import paged_kv_gqa_13_gb300 as pd

    code = {"f16": pd.PD_F16, "bf16": pd.PD_BF16}[dtype]
    want = pd.PD_KERNEL_FP8_TENSOR_CORES if Hq // Hk >= 4 else pd.PD_KERNEL_CUDA_CORES
    assert pd.pd_decode_kernel_kind(Hq, Hk, 128, code, True) == want
    rng = np.random.default_rng(341)
    lens = rng.integers(0, 70, size=600)
    w = wl.make_paged("fp8_big_batch", dtype, lens, Hq, Hk, 128, 16, seed=342)
    dev = Fp8Device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), dtype, "fp8 batch 600")
    assert pd.pd_read_device_flags(dev.ws) == 0


@pytest.mark.parametrize("lead,trail", [(0, 37), (45, 0), (29, 64)])
def test_fp8_indices_entries_that_no_request_lists(lead, trail):
    """`indices` may hold entries outside [indptr[0], indptr[batch]): the E4M3
    tensor-core kernel's walk skips those positions and still meets every
    listed page once."""
    import dataclasses

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("fp8_unlisted", "bf16", [2400, 2390, 2401, 2397], 32, 8, 128, 16, seed=343)
    t = w.table
    filler = t.indices[:max(lead, trail)]  # valid page ids that no request lists here
    t2 = dataclasses.replace(t, indices=np.concatenate([filler[:lead], t.indices, filler[:trail]]).astype(np.int32),
                             indptr=(t.indptr + lead).astype(np.int32))
    dev = Fp8Device(w)
    dev.set_table(t2)
    o, lse = dev.decode()
    assert pd.pd_read_device_flags(dev.ws) == 0
    compare(o, lse, *dev.oracle_decode(), "bf16", f"fp8, {lead} leading, {trail} trailing unlisted entries")


@pytest.mark.parametrize("tcgen05", [False, True])
def test_fp8_decode_replays_from_a_cuda_graph(tcgen05):
    """The E4M3 decode (either tensor-core kernel) captured once into a CUDA
    graph and replayed: bit-identical to the direct call, and it reads new q
    and new page contents in place."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("fp8_graph", "bf16", [700, 1, 2400, 33, 1600], 32, 8, 128, 16, seed=344)
    pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TCGEN05 if tcgen05 else pd.PD_KERNEL_FP8_TENSOR_CORES)
    try:
        dev = Fp8Device(w)  # the workspace size follows the selected kernel
        want = pd.PD_KERNEL_FP8_TCGEN05 if tcgen05 else pd.PD_KERNEL_FP8_TENSOR_CORES
        assert pd.pd_decode_kernel_kind(32, 8, 128, pd.PD_BF16, True) == want
        ref_o, ref_lse = (x.clone() for x in dev.decode())  # the first call plans the shape
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dev.decode()
        for _ in range(2):
            dev.o.fill_(7)
            dev.lse.fill_(7)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(dev.o.view(torch.int16), ref_o.view(torch.int16))
            assert torch.equal(dev.lse, ref_lse)
        q2 = wl.normal(w.q.shape, w.dtype, wl.stream_key(w.seed + 5, "q"))
        dev.q.copy_(to_dev(q2, w.dtype))
        w.q = q2
        dev.k8 ^= np.uint8(0x80)  # every K value negated (NaN codes in unused rows stay NaN)
        dev.k.copy_(torch.from_numpy(dev.k8).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert pd.pd_read_device_flags(dev.ws) == 0
        compare(dev.o, dev.lse, *dev.oracle_decode(), "bf16", "fp8 graph replay, new q and K codes")
    finally:
        pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TENSOR_CORES)
