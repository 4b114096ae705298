"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects malformed arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedecode.h")


def _declared():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for n in ("pd_paged_decode", "pd_paged_append", "pd_contiguous_decode", "pd_merge_states",
              "pd_paged_decode_workspace_bytes", "pd_last_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import paged_kv_gqa_13_gb300 as pd

    lib = ctypes.CDLL(pd.LIBRARY_PATH)
    for name in _declared():
        assert hasattr(lib, name), f"{name} not exported"
    assert set(_declared()) == set(pd.EXPORTED)
    assert pd.pd_version() == 1


FAKE = 1 << 20  # an aligned address that is never dereferenced: every call below fails its checks first


def _decode(**kw):
    import paged_kv_gqa_13_gb300 as pd

    args = dict(q=FAKE, k=FAKE, v=FAKE, indices=FAKE, indptr=FAKE, lpl=FAKE, o=FAKE, lse=FAKE, batch=2,
                hq=8, hk=2, d=128, p=16, pages=10, nidx=4, scale=0.1, dtype=pd.PD_BF16, ws=FAKE,
                wsb=1 << 20, stream=None)
    args.update(kw)
    return pd._lib.pd_paged_decode(*args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(batch=0), 1), (dict(hq=0), 1), (dict(hk=-1), 1), (dict(p=0), 1), (dict(pages=0), 1),
    (dict(nidx=-1), 1), (dict(hq=9), 1), (dict(d=96), 2), (dict(d=512), 2), (dict(dtype=7), 2),
    (dict(q=None), 1), (dict(lse=None), 1), (dict(indices=None), 1), (dict(o=FAKE + 8), 2),
    (dict(k=FAKE + 4), 2), (dict(indptr=FAKE + 2), 2), (dict(scale=float("nan")), 1),
])
def test_paged_decode_rejects_bad_arguments(kw, status):
    import paged_kv_gqa_13_gb300 as pd

    assert _decode(**kw) == status
    assert pd.pd_last_error_string() != ""


def test_indices_may_be_null_when_empty():
    import paged_kv_gqa_13_gb300 as pd

    # Passes the argument checks; then stops at the device query (no GPU) or at the
    # too-small fake workspace (GPU present). Nothing is launched either way.
    st = _decode(indices=None, nidx=0, wsb=4096)
    assert st in (pd.PD_ERR_CUDA, pd.PD_ERR_WORKSPACE)


def test_contiguous_and_append_and_merge_reject_bad_arguments():
    import paged_kv_gqa_13_gb300 as pd

    L = pd._lib
    # valid_kv_len > max_kv_len
    assert L.pd_contiguous_decode(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 128, 10, 11, 0.1, pd.PD_F16, FAKE,
                                  1 << 20, None) == pd.PD_ERR_INVALID
    assert L.pd_contiguous_decode(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 80, 10, 5, 0.1, pd.PD_F16, FAKE,
                                  1 << 20, None) == pd.PD_ERR_UNSUPPORTED
    assert L.pd_paged_append(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 128, 16, 10, 4, pd.PD_F16, FAKE,
                             256, None) == pd.PD_ERR_INVALID
    assert L.pd_paged_append(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 16, 10, 4, pd.PD_F16, None,
                             0, None) == pd.PD_ERR_WORKSPACE
    assert L.pd_paged_append(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 16, 10, 4, pd.PD_F16, FAKE,
                             16, None) == pd.PD_ERR_WORKSPACE
    # contiguous append: position outside [0, max_kv_len), bad head_dim, null cache
    assert L.pd_contiguous_append(FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 40, 40, pd.PD_F16, None) == pd.PD_ERR_INVALID
    assert L.pd_contiguous_append(FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 40, -1, pd.PD_F16, None) == pd.PD_ERR_INVALID
    assert L.pd_contiguous_append(FAKE, FAKE, FAKE, FAKE, 2, 2, 96, 40, 3, pd.PD_F16, None) == pd.PD_ERR_UNSUPPORTED
    assert L.pd_contiguous_append(FAKE, FAKE, None, FAKE, 2, 2, 128, 40, 3, pd.PD_F16, None) == pd.PD_ERR_INVALID
    assert L.pd_merge_states(FAKE, FAKE, 0, 4, 128, FAKE, None, pd.PD_F32, None) == pd.PD_ERR_INVALID
    assert L.pd_merge_states(FAKE, FAKE, 2, 4, 100, FAKE, None, pd.PD_F32, None) == pd.PD_ERR_UNSUPPORTED
    assert L.pd_copy_bytes(FAKE, FAKE, 10, None) == pd.PD_ERR_UNSUPPORTED
    assert L.pd_workspace_init(FAKE, 8, None) == pd.PD_ERR_WORKSPACE


def test_a_c_program_compiles_links_and_runs_against_the_header(tmp_path):
    """The boundary is usable from plain C: a C11 translation unit includes the
    header, takes the address of every declared entry point, links against the
    built library and calls the two entry points that need no device."""
    import shutil
    import subprocess

    import paged_kv_gqa_13_gb300 as pd

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = _declared()
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include <stdio.h>\n#include "pagedecode.h"\n'
        "int main(void) {\n"
        "    void (*fns[])(void) = {" + ", ".join(f"(void (*)(void)){n}" for n in names) + "};\n"
        "    int nonnull = 0;\n"
        "    for (unsigned i = 0; i < sizeof fns / sizeof fns[0]; ++i) nonnull += fns[i] != 0;\n"
        "    printf(\"%d %d %s\\n\", nonnull, pd_version(), pd_last_error_string() ? \"str\" : \"null\");\n"
        "    return 0;\n}\n")
    libdir = os.path.dirname(pd.LIBRARY_PATH)
    exe = tmp_path / "use_abi"
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lpagedecode", f"-Wl,-rpath,{libdir}",
                    "-Wl,--unresolved-symbols=ignore-in-shared-libs", "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    env = dict(os.environ)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, env=env).stdout.split()
    assert out == [str(len(names)), "1", "str"]


def _expected_kind(hq, hk, d, dtype, fp8, tcgen05=False):
    """The dispatch rule, written out: the group is cut into the fewest equal
    tiles of at most 8 heads, padded to 1, 2, 4 or 8; 16-bit tiles of 4 or 8
    run on tensor cores; over E4M3 pools only at head_dim 128 or 256, and, when
    the tcgen05 kernel is selected, with bf16 q, groups of exactly 4 and an
    even number of kv heads at head_dim 128 on that kernel."""
    import paged_kv_gqa_13_gb300 as pd

    if hq <= 0 or hk <= 0 or hq % hk or d not in (64, 128, 256) or (fp8 and dtype == pd.PD_F32):
        return pd.PD_KERNEL_NONE
    g = hq // hk
    tiles = next(t for t in range(1, g + 1) if g % t == 0 and g // t <= 8)
    pad = 1 << (g // tiles - 1).bit_length()
    if fp8:
        if tcgen05 and d == 128 and dtype == pd.PD_BF16 and g == 4 and hk % 2 == 0:
            return pd.PD_KERNEL_FP8_TCGEN05
        return pd.PD_KERNEL_FP8_TENSOR_CORES if (d >= 128 and pad >= 4) else pd.PD_KERNEL_CUDA_CORES
    return pd.PD_KERNEL_TENSOR_CORES if (dtype != pd.PD_F32 and pad >= 4) else pd.PD_KERNEL_CUDA_CORES


def test_decode_kernel_kind_follows_the_dispatch_rule():
    """pd_decode_kernel_kind is a host-side lookup (no device needed); the GPU
    tests use it to check which kernel their shapes reach."""
    import paged_kv_gqa_13_gb300 as pd

    k = pd.pd_decode_kernel_kind
    # the shapes of the workloads
    assert k(32, 8, 128, pd.PD_BF16) == pd.PD_KERNEL_TENSOR_CORES        # Llama-3-8B, group 4
    assert k(64, 8, 128, pd.PD_BF16) == pd.PD_KERNEL_TENSOR_CORES        # 70B, group 8
    assert k(16, 16, 256, pd.PD_F16) == pd.PD_KERNEL_CUDA_CORES          # MHA D 256
    assert k(8, 2, 64, pd.PD_F32) == pd.PD_KERNEL_CUDA_CORES             # tiny f32
    assert k(32, 8, 128, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES
    assert k(32, 8, 64, pd.PD_BF16, True) == pd.PD_KERNEL_CUDA_CORES     # E4M3 at D 64
    assert k(8, 3, 128, pd.PD_F16) == pd.PD_KERNEL_NONE                  # not a multiple
    assert k(8, 2, 96, pd.PD_F16) == pd.PD_KERNEL_NONE                   # head_dim
    assert k(8, 2, 128, pd.PD_F32, True) == pd.PD_KERNEL_NONE            # E4M3 takes 16-bit q
    for dtype in (pd.PD_F32, pd.PD_F16, pd.PD_BF16):
        for d in (64, 96, 128, 256):
            for hk in (1, 2, 8):
                for g in range(1, 25):
                    for fp8 in (False, True):
                        assert k(g * hk, hk, d, dtype, fp8) == _expected_kind(g * hk, hk, d, dtype, fp8), \
                            (g, hk, d, dtype, fp8)


def test_fp8_kernel_selection_changes_the_dispatch_only_where_both_kernels_apply():
    """pd_select_fp8_kernel picks the tcgen05 E4M3 kernel for bf16 q, groups of
    exactly 4, an even number of kv heads and head_dim 128; every other shape
    keeps its kernel. Host-side only."""
    import paged_kv_gqa_13_gb300 as pd

    k = pd.pd_decode_kernel_kind
    try:
        pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TCGEN05)
        assert k(32, 8, 128, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TCGEN05      # Llama-3-8B shape
        assert k(64, 8, 128, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES  # group 8
        assert k(32, 8, 128, pd.PD_F16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES   # f16 q
        assert k(12, 3, 128, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES  # odd number of kv heads
        assert k(32, 8, 256, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES  # head_dim 256
        assert k(32, 8, 128, pd.PD_BF16) == pd.PD_KERNEL_TENSOR_CORES            # 16-bit pools unchanged
        for dtype in (pd.PD_F16, pd.PD_BF16):
            for d in (64, 128, 256):
                for hk in (1, 2, 3, 8):
                    for g in range(1, 13):
                        for fp8 in (False, True):
                            assert k(g * hk, hk, d, dtype, fp8) == _expected_kind(g * hk, hk, d, dtype, fp8, True), \
                                (g, hk, d, dtype, fp8)
        with pytest.raises(pd.PagedecodeError):
            pd.pd_select_fp8_kernel(pd.PD_KERNEL_TENSOR_CORES)
    finally:
        pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TENSOR_CORES)
    assert k(32, 8, 128, pd.PD_BF16, True) == pd.PD_KERNEL_FP8_TENSOR_CORES
