"""GPU parity of the CUDA-core decode kernel (`decode_kernel`) at every class
of page size, through the C ABI, against the CPU oracle.

The CUDA-core kernel serves f32 at every group and 16-bit tiles of 1 or 2 q
heads per kv head (the MHA shape), plus E4M3 pools outside the E4M3
tensor-core kernel's shapes. Its pipeline stage holds kRC = 4096 bytes of K
rows (and as many of V): 4 rows at head_dim 256 f32, 8 at 128 f32 or 256
16-bit, 16 at 64 f32 or 128 16-bit, 32 at 64 16-bit; for E4M3 pools 32 rows at
128 and 64 at 64. A page is copied in chunks of at most kRC rows, so the page
sizes below take every chunk path: one-row pages (one row per chunk), pages
shorter than a stage (4, 8), pages that are whole multiples of a stage (32,
64), and pages that end in a partial chunk (100 = 12 x 8 + 4 at 8 rows per
stage). Any page size and any last_page_len in 0..page_size are legal
(batch_paged_decode.rs, module doc, "Layout").

Each test first checks that its shape really dispatches to the CUDA-core
kernel, with the rule written out here and with the library's own answer
(pd_decode_kernel_kind), so that a change of dispatch cannot silently move
the coverage to another kernel.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.gpu_helpers import DeviceWorkload, Fp8Device, compare, to_dev, to_host_raw

pytestmark = pytest.mark.gpu

PAGE_SIZES = [1, 4, 8, 32, 64, 100]
CODE = {"f32": 0, "f16": 1, "bf16": 2}


def expected_kernel(hq: int, hk: int, head_dim: int, dtype: str, fp8: bool = False) -> str:
    """The dispatch rule: the group is cut into the fewest equal tiles of at
    most 8 heads, each padded to a power of two; 16-bit tiles of 4 or 8 run on
    tensor cores; over E4M3 pools only at head_dim 128 or 256."""
    g = hq // hk
    tiles = next(t for t in range(1, g + 1) if g % t == 0 and g // t <= 8)
    pad = 1 << (g // tiles - 1).bit_length()
    if fp8:
        return "fp8_tensor_cores" if (head_dim >= 128 and pad >= 4) else "cuda_cores"
    return "tensor_cores" if (dtype != "f32" and pad >= 4) else "cuda_cores"


def assert_cuda_cores(hq, hk, head_dim, dtype, fp8=False):
    import paged_kv_gqa_13_gb300 as pd

    assert expected_kernel(hq, hk, head_dim, dtype, fp8) == "cuda_cores"
    assert pd.pd_decode_kernel_kind(hq, hk, head_dim, CODE[dtype], fp8) == pd.PD_KERNEL_CUDA_CORES


def lens_for(page_size: int):
    """Ragged lengths: empty, one row, exact page multiples, a partly filled
    last page, and lengths that end inside a chunk."""
    P = page_size
    return [0, 1, P, 2 * P, 3 * P + max(1, P // 3), 333, 17, 5 * P - 1]


def _decode_vs_oracle(w):
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    compare(o, lse, *oracle.paged_decode_workload(w), w.dtype, w.name)
    assert dw.flags() == 0


@pytest.mark.parametrize("page_size", PAGE_SIZES)
@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("hq,hk", [(4, 4), (8, 4), (8, 2)])  # groups 1, 2, 4
def test_f32_every_group(page_size, head_dim, hq, hk):
    assert_cuda_cores(hq, hk, head_dim, "f32")
    w = wl.make_paged(f"cc_f32_{hq}_{hk}_{head_dim}_p{page_size}", "f32", lens_for(page_size), hq, hk, head_dim,
                      page_size, seed=500 + page_size + head_dim + 7 * hq + hk)
    _decode_vs_oracle(w)


@pytest.mark.parametrize("page_size", PAGE_SIZES)
@pytest.mark.parametrize("head_dim", [128, 256])
@pytest.mark.parametrize("hq,hk", [(8, 8), (16, 8)])  # groups 1, 2
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_16bit_groups_of_one_and_two(page_size, head_dim, hq, hk, dtype):
    assert_cuda_cores(hq, hk, head_dim, dtype)
    w = wl.make_paged(f"cc_{dtype}_{hq}_{hk}_{head_dim}_p{page_size}", dtype, lens_for(page_size), hq, hk,
                      head_dim, page_size, seed=600 + page_size + head_dim + 7 * hq + (dtype == "bf16"))
    _decode_vs_oracle(w)


@pytest.mark.parametrize("dtype,hq,hk,head_dim,page_size", [
    ("f32", 8, 4, 128, 4),     # group 2, four-row pages
    ("f32", 16, 4, 64, 1),     # group 4, one-row pages
    ("f16", 16, 16, 256, 4),   # MHA D 256
    ("bf16", 16, 8, 128, 1),   # group 2, one-row pages
])
def test_long_shares_take_tails(dtype, hq, hk, head_dim, page_size):
    """Enough positions that every warp's share holds at least 12 (one- and
    four-row pages), so the last eighth of each share is handed out at run time
    and long requests are split over many warps."""
    import paged_kv_gqa_13_gb300 as pd
    import torch

    assert_cuda_cores(hq, hk, head_dim, dtype)
    w = wl.make_paged(f"cc_tails_{dtype}_{hq}_{hk}_{head_dim}_p{page_size}", dtype,
                      [1, 9000, 6003, 77, 4 * page_size, 0], hq, hk, head_dim, page_size,
                      seed=700 + page_size + head_dim + hq)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = hq // hk
    head_tiles = next(t for t in range(1, g + 1) if g % t == 0 and g // t <= 8)
    positions = hk * head_tiles * w.table.num_indices
    assert positions >= 12 * 8 * sms, "the shape must give shares of at least 12 positions"
    dw = DeviceWorkload(w)
    o, lse = dw.decode()
    o1, l1 = o.clone(), lse.clone()
    compare(o, lse, *oracle.paged_decode_workload(w), dtype, w.name)
    o2, l2 = dw.decode()  # the tail counters are back at zero: a repeat is bit-identical
    raw = (lambda x: x) if dtype == "f32" else (lambda x: x.view(torch.int16))
    assert torch.equal(raw(o1), raw(o2)) and torch.equal(l1, l2)
    assert dw.flags() == 0
    assert pd.pd_read_device_flags(dw.ws) == 0


@pytest.mark.parametrize("page_size", [1, 8, 100])
@pytest.mark.parametrize("dtype,hq,hk,head_dim", [("bf16", 16, 8, 128),   # group 2, 32 rows per stage
                                                   ("f16", 32, 8, 64)])   # group 4 at D 64, 64 rows per stage
def test_e4m3_cuda_core_variant(page_size, dtype, hq, hk, head_dim):
    assert_cuda_cores(hq, hk, head_dim, dtype, fp8=True)
    w = wl.make_paged(f"cc_e4m3_{dtype}_{hq}_{hk}_{head_dim}_p{page_size}", dtype, lens_for(page_size), hq, hk,
                      head_dim, page_size, seed=800 + page_size + head_dim)
    dev = Fp8Device(w)
    o, lse = dev.decode()
    compare(o, lse, *dev.oracle_decode(), dtype, w.name)
    import paged_kv_gqa_13_gb300 as pd

    assert pd.pd_read_device_flags(dev.ws) == 0


@pytest.mark.parametrize("page_size", [8, 32])
@pytest.mark.parametrize("dtype,hq,hk,head_dim", [("f32", 16, 4, 128), ("f16", 16, 16, 256), ("bf16", 16, 8, 128)])
def test_fused_append_decode_on_cuda_cores(page_size, dtype, hq, hk, head_dim):
    """pd_paged_append_decode per step: the pool bit for bit as the oracle's
    append leaves it, o and lse as the oracle decodes it, and both bitwise
    equal to pd_paged_append followed by pd_paged_decode."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    assert_cuda_cores(hq, hk, head_dim, dtype)
    steps = 3
    lens = [0, page_size - 1, page_size, 1, 2 * page_size - 1, 1500, 3]
    w = wl.make_paged(f"cc_fused_{dtype}_{hq}_{hk}_p{page_size}", dtype, lens, hq, hk, head_dim, page_size,
                      seed=900 + page_size + hq, extra_rows=steps, append_steps=steps)
    fused, split = DeviceWorkload(w), DeviceWorkload(w)
    k_host, v_host = w.k_data.copy(), w.v_data.copy()
    bits = np.uint32 if dtype == "f32" else np.uint16
    raw = (lambda x: x) if dtype == "f32" else (lambda x: x.view(torch.int16))
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
        assert torch.equal(raw(fused.o), raw(o2)), f"fused o differs from append + decode, step {step}"
        assert torch.equal(fused.lse, l2), f"fused lse differs from append + decode, step {step}"
    assert fused.flags() == 0 and split.flags() == 0
