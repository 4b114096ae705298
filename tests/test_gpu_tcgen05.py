"""GPU parity for the tcgen05 E4M3 decode kernel (pd_select_fp8_kernel), which
serves bf16 q with groups of exactly 4 q heads and an even number of kv heads
at head_dim 128, kv heads in pairs: every output against the oracle's FP8
decode, over page sizes that give one 16-row box per page (1, 3, 8, 16) and
several (32, 100), ragged and empty requests, page ids that no request lists,
appends between decodes, the full Llama-shaped batch, a seeded random sweep
and a bounded wait that runs out."""
import time

import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import Fp8Device, compare, to_dev
from tests.test_gpu_random import with_unlisted_entries

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 100, 3000, 33, 64, 65, 511]


@pytest.fixture(autouse=True)
def tcgen05_kernel():
    import paged_kv_gqa_13_gb300 as pd

    pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TCGEN05)
    try:
        yield
    finally:
        pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TENSOR_CORES)


def torch_equal(a, b) -> bool:
    import torch

    return bool(torch.equal(a, b))


def _device(w):
    import paged_kv_gqa_13_gb300 as pd

    assert pd.pd_decode_kernel_kind(w.num_qo_heads, w.num_kv_heads, w.head_dim, pd.PD_BF16, True) == \
        pd.PD_KERNEL_FP8_TCGEN05
    return Fp8Device(w)


@pytest.mark.parametrize("Hq,Hk", [(32, 8), (8, 2), (16, 4)])
@pytest.mark.parametrize("P", [1, 3, 8, 16, 32, 100])
def test_tcgen05_decode_matches_oracle(Hq, Hk, P):
    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged(f"tc_{Hq}_{Hk}_{P}", "bf16", LENS, Hq, Hk, 128, P, seed=700 + Hq + P)
    dev = _device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", f"tcgen05 {Hq}/{Hk} page {P}")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_tcgen05_unlisted_page_ids_and_repeat_calls():
    """Entries outside [indptr[0], indptr[batch]) are skipped; a second call on
    the same workspace gives the same bits."""
    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("tc_unlisted", "bf16", [5, 300, 0, 47, 1200], 32, 8, 128, 16, seed=731, pool_slack=0.3)
    dev = _device(w)
    t = with_unlisted_entries(w, 3, 5)
    dev.set_table(t)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", "tcgen05 unlisted entries")
    first = (o.clone(), lse.clone())
    o2, lse2 = dev.decode()
    assert torch_equal(o2, first[0]) and torch_equal(lse2, first[1])
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_tcgen05_append_then_decode():
    import paged_kv_gqa_13_gb300 as pd

    steps = 3
    w = wl.make_paged("tc_append", "bf16", [0, 15, 16, 31, 200], 32, 8, 128, 16, seed=741, extra_rows=steps,
                      append_steps=steps)
    dev = _device(w)
    t = w.table
    for step in range(steps):
        t = wl.table_after_append(t)
        kn, vn = w.new_rows(step)
        dev.set_table(t)
        pd.pd_paged_append_fp8(to_dev(kn, "bf16"), to_dev(vn, "bf16"), dev.ksd, dev.vsd, dev.k, dev.v, dev.ind,
                               dev.ptr, dev.lpl, dev.ws)
        oracle.paged_append_fp8(kn, vn, dev.ks, dev.vs, dev.k8, dev.v8, t.indices, t.indptr, t.last_page_len, "bf16")
        o, lse = dev.decode()
        compare(o, lse, *dev.oracle_decode(), "bf16", f"tcgen05 step {step}")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_tcgen05_full_llama3_8b_e4m3_pool():
    import paged_kv_gqa_13_gb300 as pd

    w = wl.llama3_8b_bf16()
    dev = _device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", w.name + " e4m3 tcgen05")
    assert pd.pd_read_device_flags(dev.ws) == 0


@pytest.mark.parametrize("seed", list(range(5000, 5024)))
def test_tcgen05_random(seed):
    import paged_kv_gqa_13_gb300 as pd

    rng = np.random.default_rng(seed)
    hk = int(rng.choice([2, 4, 8]))
    page = int(rng.choice([1, 3, 8, 16, 16, 16, 32, 48, 100, 128]))
    batch = int(rng.choice([1, 3, 17, 64, 130, 513, 600]))
    lens = np.clip(np.rint(np.exp(rng.normal(np.log(300), 1.3, size=batch))), 0, 20000).astype(np.int64)
    forced = [0, 1, page, 2 * page, 3 * page + 1]
    lens[: min(batch, len(forced))] = forced[: min(batch, len(forced))]
    while lens.sum() * hk > 300_000:
        lens = lens // 2
    rng.shuffle(lens)
    w = wl.make_paged(f"tcrand{seed}", "bf16", lens, 4 * hk, hk, 128, page, seed=seed)
    dev = _device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", f"seed {seed}: {4 * hk}/{hk} page {page} batch {batch}")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_tcgen05_wait_timeout_sets_the_flag_and_returns():
    """The injected missing bytes make the first stage's wait run out: the flag
    is set, every role stops within its bounded waits, the tensor memory is
    released, and the next call is exact again."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("tc_timeout", "bf16", [40, 300, 17, 1000], 32, 8, 128, 16, seed=751)
    dev = _device(w)
    dev.decode()
    torch.cuda.synchronize()
    assert pd.pd_read_device_flags(dev.ws) == 0
    pd.pd_test_inject_wait_timeout(16)
    try:
        t0 = time.perf_counter()
        dev.decode()
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        pd.pd_test_inject_wait_timeout(0)
    assert pd.pd_read_device_flags(dev.ws) & pd.PD_FLAG_WAIT_TIMEOUT
    assert 1.5 < elapsed < 30.0, elapsed
    pd.pd_workspace_init(dev.ws)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), "bf16", "tcgen05 after timeout")
    assert pd.pd_read_device_flags(dev.ws) == 0


def test_tcgen05_workspace_sizes_follow_the_selection():
    """The two E4M3 kernels partition the work differently, so their workspace
    sizes differ; a workspace sized for one and too small for the other is
    rejected with an error, never written past its end."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged("tc_ws", "bf16", [100, 2000, 37, 512], 32, 8, 128, 16, seed=761)
    ws_tc = pd.pd_paged_decode_fp8_workspace_bytes(w.batch, 32, 8, 128, pd.PD_BF16)
    pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TENSOR_CORES)
    ws_mma = pd.pd_paged_decode_fp8_workspace_bytes(w.batch, 32, 8, 128, pd.PD_BF16)
    assert ws_tc > 0 and ws_mma > 0 and ws_tc != ws_mma
    dev = Fp8Device(w)  # sized for the mma.sync kernel
    small, large = (dev.ws, None) if ws_mma < ws_tc else (None, dev.ws)
    pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TCGEN05)
    if small is not None:
        with pytest.raises(pd.PagedecodeError):
            dev.decode()
    else:
        o, lse = dev.decode()  # a larger workspace than needed is fine
        compare(o, lse, *dev.oracle_decode(), "bf16", "tcgen05 with the mma.sync workspace")
        assert pd.pd_read_device_flags(large) == 0
    torch.cuda.synchronize()
