"""A bounded wait that runs out: the kernel reports it in the status word and
returns, and the GPU context stays usable. The missing bytes are injected on
the host (pd_test_inject_wait_timeout); nothing traps, faults or hangs."""
import time

import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,dtype,Hq,Hk", [
    ("CUDA cores", "bf16", 32, 8),
    ("tensor cores", "bf16", 64, 8),
    ("E4M3 tensor cores", "bf16", 32, 8),
])
def test_wait_timeout_sets_the_flag_and_returns(kind, dtype, Hq, Hk):
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w = wl.make_paged(f"timeout_{Hq}", dtype, [40, 300, 17, 1000], Hq, Hk, 128, 16, seed=400 + Hq)
    if kind.startswith("E4M3"):
        from tests.test_gpu_fp8 import Fp8Device

        dev = Fp8Device(w)
        run, flags, ws = dev.decode, (lambda: pd.pd_read_device_flags(dev.ws)), dev.ws
        ref = dev.oracle_decode
    else:
        dev = DeviceWorkload(w)
        run, flags, ws = dev.decode, dev.flags, dev.ws
        ref = lambda: oracle.paged_decode_workload(w)  # noqa: E731
    run()
    torch.cuda.synchronize()
    assert flags() == 0
    pd.pd_test_inject_wait_timeout(16)
    try:
        t0 = time.perf_counter()
        run()
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        pd.pd_test_inject_wait_timeout(0)
    assert flags() & pd.PD_FLAG_WAIT_TIMEOUT, kind
    assert 1.5 < elapsed < 30.0, elapsed  # the 2 s limit, not a hang
    # the context is usable and the next call is exact again
    pd.pd_workspace_init(ws)
    o, lse = run()
    compare(o, lse, *ref(), dtype, kind + " after timeout")
    assert flags() == 0


def test_inject_rejects_bad_sizes():
    import paged_kv_gqa_13_gb300 as pd

    for bad in (-16, 8, 1 << 21):
        with pytest.raises(pd.PagedecodeError):
            pd.pd_test_inject_wait_timeout(bad)
    pd.pd_test_inject_wait_timeout(0)
