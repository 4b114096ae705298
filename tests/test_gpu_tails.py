"""Dynamic share tails of the tensor-core decode: shapes with enough positions
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
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(lse, l1)
    assert _counters(dw.ws) == [0, 0]
    compare(o1, l1, *oracle.paged_decode_workload(w), w.dtype, "tails")
