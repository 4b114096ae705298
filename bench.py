"""Benchmark of batched paged-KV GQA decode on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step is one batched paged-decode call (decode kernel + merge kernel; for
the append workload, an append then a decode) over the workload's batch,
inputs resident in HBM. L2 is flushed between timed steps, outside the timed
events. Prints one JSON line: achieved HBM TB/s = (K+V+q+o bytes) / device
time per call, with the roofline of the decode kernel, the CPU oracle timed on
the host as a reported baseline, an end-to-end figure through the C ABI with
host buffers, and SM clocks sampled during the run.

--impl reference times the CPU oracle (the reference arm: there is no
runnable reference implementation) on a bounded sample of the same workload.
Under torchrun every rank runs its own replica on its own GPU (the decode has
no exchange step); rank 0 prints.

On one GPU the line also carries `per_config`: the long-context batch (paged,
contiguous and token-major contiguous entries), the ragged 70B-shaped batch,
the MHA append + decode step and the Llama-shaped batch over an E4M3 pool,
each timed the same way in the same process after the headline workload
(--no-per-config skips them).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM TB/s (% of GB300 peak) and us per batched paged-decode call"
UNIT = "TB/s"
DEFAULT_CONFIG = "llama3_8b"
L2_FLUSH_BYTES = 512 << 20
KERNEL_SOURCES = ["paged_kv_gqa_13_gb300/csrc/" + f for f in
                  ("pd_device.cuh", "pd_walk.cuh", "pd_decode.cuh", "pd_decode_mma.cuh", "pd_decode_fp8.cuh",
                   "pd_decode_tc.cuh", "pd_merge.cuh")]


def kernel_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def workload_key(w, mode: str) -> str:
    """The workload column of profiles/dram_traffic.txt: the workload's name, and its entry."""
    return w.name + {"contiguous": "/contiguous", "contiguous_nhd": "/nhd", "paged_fp8": "/e4m3"}.get(mode, "")


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_sha()
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            if parts[2] == sha:
                return int(parts[3])
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle samples while the benchmark runs.

    nvidia-smi runs as its own process and writes its samples (each with its
    own timestamp) to a file, which is read after the run: no thread of this
    process competes with the launch loop while it is timed."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import tempfile

        self.marks = {}
        fd, self.path = tempfile.mkstemp(prefix="pd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index), "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, name):
        self.marks[name] = time.time()

    @staticmethod
    def _when(stamp: str):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self) -> dict:
        if self.proc is None:
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        samples = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    samples.append((self._when(parts[0]), parts[1:]))
        os.unlink(self.path)
        t0, t1 = self.marks.get("timed_start", 0), self.marks.get("timed_end", 1e30)
        timed = [p for (t, p) in samples if t is not None and t0 <= t <= t1]
        window = "timed region"
        if not timed:
            timed = [p for (_, p) in samples]
            window = "whole run (timed region shorter than the 100 ms sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in timed if num(p[1]) is not None]
        mx = [num(p[2]) for p in timed if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in timed for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(timed), "window": window}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (libnvidia-ml, read-only
    queries) every ~2 ms while the timed steps run: the timed region of one
    workload is a few tens of milliseconds, shorter than nvidia-smi's sampling
    period. The thread only starts once every timed step has been queued (the
    host is waiting on the device), so it does not delay the launches."""

    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL = 0x4, 0x8, 0x20, 0x40

    def __init__(self, device_index: int):
        import ctypes

        self.samples = []
        self.handle = None
        try:
            import torch

            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            pr = torch.cuda.get_device_properties(device_index)
            bus = b"%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                return
            self.lib, self.handle = lib, h
            mx = ctypes.c_uint(0)
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            self.handle = None

    def _poll(self, stop):
        import ctypes

        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0 and \
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            stop.wait(0.002)

    def run_while(self, wait):
        """Call wait() (a device synchronize) while sampling in a thread."""
        if self.handle is None:
            wait()
            return
        stop = threading.Event()
        t = threading.Thread(target=self._poll, args=(stop,), daemon=True)
        t.start()
        try:
            wait()
        finally:
            stop.set()
            t.join()

    def summary(self) -> dict | None:
        if self.handle is None or not self.samples:
            return None
        names = [(self.HW_SLOWDOWN, "hw_slowdown"), (self.HW_THERMAL, "hw_thermal_slowdown"),
                 (self.SW_THERMAL, "sw_thermal_slowdown"), (self.SW_POWER_CAP, "sw_power_cap")]
        reasons = sorted({n for (_, r) in self.samples for (bit, n) in names if r & bit})
        return {"sm_mhz": statistics.median(m for (m, _) in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "window": "timed region (NVML, every ~2 ms)"}


# ---------------------------------------------------------------- workloads

def load_workload(name: str, rank: int = 0):
    import workloads as wl

    if name == "long_context_contiguous":
        return wl.long_context_f16(seed=1002 + 100 * rank), "contiguous"
    if name == "long_context_nhd":
        return wl.long_context_f16(seed=1002 + 100 * rank), "contiguous_nhd"
    if name == "llama3_8b_fp8":
        return wl.llama3_8b_bf16(seed=1001 + 100 * rank), "paged_fp8"
    return wl.CONFIGS[name](seed=wl.CONFIGS[name].__defaults__[0] + 100 * rank), "paged"


def decode_kernel_name(w, mode: str = "paged") -> str:
    """The decode kernel the library runs for this workload (its own host-side
    lookup, pd_decode_kernel_kind)."""
    import paged_kv_gqa_13_gb300 as pd

    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[w.dtype]
    kind = pd.pd_decode_kernel_kind(w.num_qo_heads, w.num_kv_heads, w.head_dim, code, mode == "paged_fp8")
    return {pd.PD_KERNEL_CUDA_CORES: "decode_kernel", pd.PD_KERNEL_TENSOR_CORES: "decode_mma_kernel",
            pd.PD_KERNEL_FP8_TENSOR_CORES: "decode_fp8_mma_kernel",
            pd.PD_KERNEL_FP8_TCGEN05: "decode_tc_fp8_kernel"}[kind]


def algorithmic_bytes(w, table=None, mode: str = "paged") -> int:
    """K and V rows read (one byte per element for E4M3 pools, plus the two
    scale vectors), q read and o written."""
    if mode == "paged_fp8":
        import workloads as wl

        return w.kv_bytes(table) // wl.ELEM_BYTES[w.dtype] + 2 * 4 * w.num_kv_heads + w.qo_bytes()
    return w.kv_bytes(table) + w.qo_bytes()


# ---------------------------------------------------------------- GPU arm

# Extra workloads timed in the same process after the headline one (one GPU
# only): the long-context batch through the paged, the contiguous and the
# token-major contiguous entry, the ragged 70B-shaped batch, the MHA append +
# decode step, and the Llama-shaped batch over an E4M3 pool.
PER_CONFIG = ["long_context", "long_context_contiguous", "long_context_nhd", "ragged_70b", "mha_append",
              "llama3_8b_fp8"]
# Host lead before the timed steps: the stream first runs a spin kernel of
# this length, so that every timed step is already queued when the GPU
# reaches it and no host pause (GC, a thread switch) lands inside a step.
PREROLL_S = 5e-3


def to_dev(raw, dtype, device):
    import torch

    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(raw)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(raw).view(np.int16)).to(device)
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def table_dev(t, device):
    import torch

    return tuple(torch.from_numpy(x.astype(np.int32)).to(device) for x in (t.indices, t.indptr, t.last_page_len))


def setup_config(args, name: str, rank: int, dev) -> dict:
    """Device copies of one workload and its step function: the library call a
    step makes, and the algorithmic bytes per step (all kernels, and the decode
    kernel's own)."""
    import torch

    import paged_kv_gqa_13_gb300 as pd
    import workloads as wl

    w, mode = load_workload(name, rank)
    code = {"f32": pd.PD_F32, "f16": pd.PD_F16, "bf16": pd.PD_BF16}[w.dtype]
    c = {"w": w, "mode": mode, "tables": [w.table]}
    q = to_dev(w.q, w.dtype, dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.batch, w.num_qo_heads, dtype=torch.float32, device=dev)
    c.update(q=q, o=o, lse=lse)
    if mode.startswith("contiguous"):
        kc, vc, n_valid = wl.contiguous_copy(w)
        k = to_dev(kc, w.dtype, dev)
        v = to_dev(vc, w.dtype, dev)
        del kc, vc
        decode = pd.pd_contiguous_decode
        if mode == "contiguous_nhd":  # token-major [batch, max_kv_len, Hk, D]
            k, v = k.transpose(1, 2).contiguous(), v.transpose(1, 2).contiguous()
            decode = pd.pd_contiguous_decode_nhd
        ws = pd.alloc_workspace(pd.pd_contiguous_decode_workspace_bytes(
            w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, code), dev)

        def step(i):
            decode(q, k, v, o, lse, n_valid, w.sm_scale, ws)
        c["bytes"] = [algorithmic_bytes(w)]
        c["decode_bytes"] = c["bytes"]
    elif mode == "paged_fp8":
        k8, v8, ks, vs = wl.fp8_pool(w)
        k, v = torch.from_numpy(k8).to(dev), torch.from_numpy(v8).to(dev)
        ksd, vsd = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
        del k8, v8
        ws = pd.alloc_workspace(pd.pd_paged_decode_fp8_workspace_bytes(
            w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, code), dev)
        ind, ptr, lpl = table_dev(w.table, dev)

        def step(i):
            pd.pd_paged_decode_fp8(q, k, v, ksd, vsd, ind, ptr, lpl, o, lse, w.sm_scale, ws)
        c["bytes"] = [algorithmic_bytes(w, mode=mode)]
        c["decode_bytes"] = c["bytes"]
    else:
        k = to_dev(w.k_data, w.dtype, dev)
        v = to_dev(w.v_data, w.dtype, dev)
        ws = pd.alloc_workspace(pd.pd_paged_decode_workspace_bytes(
            w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, code), dev)
        tables, appends = [w.table], []
        if w.append_steps:
            # append-then-decode: each step appends one row per request, then decodes
            t = w.table
            for s_ in range(w.append_steps):
                t = wl.table_after_append(t)
                tables.append(t)
                kn, vn = w.new_rows(s_)
                appends.append((to_dev(kn, w.dtype, dev), to_dev(vn, w.dtype, dev)))
            tables = tables[1:]
        dev_tables = [table_dev(t, dev) for t in tables]
        fused = args.append == "fused"

        # Step i uses table i mod steps. Repeating the sequence rewrites the same
        # rows with the same bytes, and a decode never reads rows appended later,
        # so the cache needs no reset between repetitions.
        def step(i):
            if w.append_steps:
                j = i % w.append_steps
                ind, ptr, lpl = dev_tables[j]
                kn, vn = appends[j]
                if fused:
                    pd.pd_paged_append_decode(q, kn, vn, k, v, ind, ptr, lpl, o, lse, w.sm_scale, ws)
                    return
                pd.pd_paged_append(kn, vn, k, v, ind, ptr, lpl, ws)
            else:
                ind, ptr, lpl = dev_tables[0]
            pd.pd_paged_decode(q, k, v, ind, ptr, lpl, o, lse, w.sm_scale, ws)
        c["tables"] = tables
        c["bytes"] = [algorithmic_bytes(w, t) for t in tables]
        c["decode_bytes"] = list(c["bytes"])
        if w.append_steps:
            ab = 2 * w.batch * w.num_kv_heads * w.head_dim * wl.ELEM_BYTES[w.dtype] * 2
            c["bytes"] = [b + ab for b in c["bytes"]]
            if fused:  # the one kernel also moves the appended rows
                c["decode_bytes"] = c["bytes"]
    c.update(k=k, v=v, ws=ws, step=step)
    return c


def time_steps(c, steps: int, warmup: int, flush_l2, stream, barrier=None, sampler=None, nvml=None) -> dict:
    """W warm-up steps, then K timed steps (one CUDA event pair each, L2
    flushed before each outside the pair), then the same K steps again with
    the library's own events around each kernel (an event between the decode
    and merge launches would serialise the pair, so they are kept out of the
    first pass)."""
    import gc

    import torch

    import paged_kv_gqa_13_gb300 as pd

    step = c["step"]
    for i in range(warmup):
        flush_l2()
        step(i)
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    preroll = int(PREROLL_S * 2.07e9)
    gc.disable()
    try:
        if sampler is not None:
            sampler.mark("timed_start")
        torch.cuda._sleep(preroll)
        for i in range(steps):
            flush_l2()  # evict K/V of the previous step from L2 (outside the timed events)
            starts[i].record(stream)
            step(warmup + i)
            ends[i].record(stream)
        if nvml is not None:
            nvml.run_while(torch.cuda.synchronize)
        else:
            torch.cuda.synchronize()
        if sampler is not None:
            sampler.mark("timed_end")
        if barrier is not None:
            barrier()
        pd.pd_profile_read()  # discard anything recorded before
        pd.pd_profile_enable(True)
        torch.cuda._sleep(preroll)
        for i in range(steps):
            flush_l2()
            step(warmup + i)
        torch.cuda.synchronize()
    finally:
        gc.enable()
        pd.pd_profile_enable(False)
    prof = pd.pd_profile_read()
    ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]

    def mean_of(xs):
        return float(np.mean([xs[(warmup + i) % len(xs)] for i in range(steps)]))
    return {"ms": ms, "ms_mean": float(np.mean(ms)), "prof": prof, "bytes_mean": mean_of(c["bytes"]),
            "decode_bytes_mean": mean_of(c["decode_bytes"])}


def kernel_roofline(c, t, peak_gbs: float) -> dict:
    prof = t["prof"]
    dec_ms = prof["decode_ms"] / max(1, prof["decode_launches"])
    achieved = t["decode_bytes_mean"] / (dec_ms * 1e-3) / 1e9 if dec_ms > 0 else None
    return {"kernel": decode_kernel_name(c["w"], c["mode"]), "achieved": achieved,
            "frac": achieved / peak_gbs if achieved else None, "kernel_us": dec_ms * 1e3,
            "merge_us": prof["merge_ms"] / max(1, prof["merge_launches"]) * 1e3,
            "append_us": (prof["append_ms"] / prof["append_launches"] * 1e3) if prof["append_launches"] else None}


def step_stats(ms) -> dict:
    us = np.asarray(ms) * 1e3
    return {"us_p10_p50_p90": [float(np.percentile(us, x)) for x in (10, 50, 90)],
            "us_p99_max": [float(np.percentile(us, 99)), float(us.max())]}


def run_e2e(c, args, dev, flush_l2, stream):
    """End to end through the C ABI with host buffers: per step, copy q and
    the page table in from pinned host memory (the library's copy kernel reads
    them there), decode with o and lse in pinned host memory (the kernels'
    stores cross to the host; no copy back)."""
    import torch

    import paged_kv_gqa_13_gb300 as pd

    w, q, o, lse, k, v, ws = c["w"], c["q"], c["o"], c["lse"], c["k"], c["v"], c["ws"]
    # One step end to end: the step's inputs (q and the page table) go in
    # from pinned host memory in one copy, and the decode writes o and lse
    # straight into pinned host memory. Pinned host memory is reachable from
    # kernels at its host address under unified addressing: the copy kernel
    # reads the ~280 KB of inputs there in ~2 us less than the copy engine's
    # ~7.5 us, and the stores save a ~7 us copy back. The KV cache is
    # resident state, like weights.
    t = c["tables"][0]
    esz = q.element_size()
    parts_in = [("q", q.numel() * esz), ("indices", 4 * t.num_indices), ("indptr", 4 * (w.batch + 1)),
                ("lpl", 4 * w.batch)]
    offs, n = {}, 0
    for name, nb in parts_in:
        offs[name] = n
        n += (nb + 15) // 16 * 16  # keep every view 16-byte aligned
    h_in = torch.empty(n, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(n, dtype=torch.uint8, device=dev)
    q_host = np.ascontiguousarray(w.q).view(np.uint8).reshape(-1)
    h_in[offs["q"]:offs["q"] + q_host.size] = torch.from_numpy(q_host)
    for name, arr in (("indices", t.indices), ("indptr", t.indptr), ("lpl", t.last_page_len)):
        b = np.ascontiguousarray(arr.astype(np.int32)).view(np.uint8).reshape(-1)
        h_in[offs[name]:offs[name] + b.size] = torch.from_numpy(b)

    def view(buf, name, nbytes, dtype, shape):
        return buf[offs[name]:offs[name] + nbytes].view(dtype).view(shape)
    qd = view(d_in, "q", q.numel() * esz, q.dtype, q.shape)
    ind_d = view(d_in, "indices", 4 * t.num_indices, torch.int32, (t.num_indices,))
    ptr_d = view(d_in, "indptr", 4 * (w.batch + 1), torch.int32, (w.batch + 1,))
    lpl_d = view(d_in, "lpl", 4 * w.batch, torch.int32, (w.batch,))
    ob = o.numel() * esz
    h_out = torch.empty(ob + 4 * lse.numel(), dtype=torch.uint8).pin_memory()
    oh = h_out[:ob].view(q.dtype).view(o.shape)
    lseh = h_out[ob:].view(torch.float32).view(lse.shape)
    es = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    host_s = []
    for i in range(args.warmup + args.steps):
        if i >= args.warmup:
            flush_l2()
            es[2 * (i - args.warmup)].record(stream)
        h0 = time.perf_counter()
        pd.pd_copy_bytes(d_in, h_in, n)
        pd.pd_paged_decode(qd, k, v, ind_d, ptr_d, lpl_d, oh, lseh, w.sm_scale, ws)
        host_s.append(time.perf_counter() - h0)
        if i >= args.warmup:
            es[2 * (i - args.warmup) + 1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([es[2 * j].elapsed_time(es[2 * j + 1]) for j in range(args.steps)]))
    # the host-resident result must be the one a device-resident decode gives
    o_dev, lse_dev = torch.empty_like(oh, device=dev), torch.empty_like(lseh, device=dev)
    pd.pd_paged_decode(qd, k, v, ind_d, ptr_d, lpl_d, o_dev, lse_dev, w.sm_scale, ws)
    torch.cuda.synchronize()
    if not (torch.equal(oh.view(torch.uint8), o_dev.cpu().view(torch.uint8)) and torch.equal(lseh, lse_dev.cpu())):
        raise RuntimeError("e2e: the decode into pinned host memory differs from the device-resident decode")
    bytes_mean = float(np.mean(c["bytes"]))
    return {"value": bytes_mean / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": int(n), "d2h_bytes_per_step": int(h_out.numel()),
            "d2h": "o and lse stored by the kernels into pinned host memory",
            "host_us_per_step": 1e6 * float(np.median(host_s[args.warmup:]))}


def run_gpu(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch

    import paged_kv_gqa_13_gb300 as pd

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    pd.pd_select_fp8_kernel(pd.PD_KERNEL_FP8_TCGEN05 if args.fp8_kernel == "tcgen05" else pd.PD_KERNEL_FP8_TENSOR_CORES)
    c = setup_config(args, args.config, rank, dev)

    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer 4x the L2 (evicts every line of the last step), then
        # read one 2x the L2 so that the dirty lines of that write are written
        # back here, not inside the next timed step: the step starts with a
        # cold, clean L2. The sum goes into a tensor allocated up front: a
        # first allocation inside the timed loop would call cudaMalloc, which
        # waits for the device and leaves the step after it without a host
        # lead (one 160 us step in 20, measured).
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_out)

    # in-process copy-kernel bandwidth (reported beside the measured peak of MEASURED_PEAKS.json)
    copy_gbs = None
    if not args.quick:
        src = torch.empty(1 << 31, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        for _ in range(3):
            pd.pd_copy_bytes(dst, src)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            pd.pd_copy_bytes(dst, src)
        e1.record()
        torch.cuda.synchronize()
        copy_gbs = 2 * src.numel() * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del src, dst

    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    entries = [x.strip() for x in visible.split(",") if x.strip()]
    sampler = ClockSampler(entries[local_rank] if local_rank < len(entries) else local_rank)
    nvml = NvmlSampler(local_rank)
    barrier = torch.distributed.barrier if world > 1 else None
    t_wall = time.perf_counter()
    t = time_steps(c, args.steps, args.warmup, flush_l2, stream, barrier, sampler, nvml)
    t_wall = time.perf_counter() - t_wall
    e2e = None
    if c["mode"] == "paged" and not c["w"].append_steps and not args.quick:
        e2e = run_e2e(c, args, dev, flush_l2, stream)
    clocks = sampler.stop()
    timed_clocks = nvml.summary()
    if timed_clocks is not None:
        timed_clocks["nvidia_smi_whole_run"] = clocks
        clocks = timed_clocks
    out = {"w": c["w"], "mode": c["mode"], "ms_mean": t["ms_mean"], "ms_all": t["ms"], "bytes_mean": t["bytes_mean"],
           "decode_bytes_mean": t["decode_bytes_mean"], "prof": t["prof"], "copy_gbs": copy_gbs, "e2e": e2e,
           "clocks": clocks, "t_wall": t_wall, "per_config": None}
    if world == 1 and args.per_config and not args.quick:
        del c
        torch.cuda.empty_cache()
        peak = measured_peaks()["hbm_gbs"]
        per = {}
        for name in PER_CONFIG:
            if name == args.config:
                continue
            pc = setup_config(args, name, rank, dev)
            tp = time_steps(pc, args.steps, args.warmup, flush_l2, stream)
            kr = kernel_roofline(pc, tp, peak)
            tbps = tp["bytes_mean"] / (tp["ms_mean"] * 1e-3) / 1e12
            per[name] = {"workload": pc["w"].name, "mode": pc["mode"], "us_per_call": tp["ms_mean"] * 1e3,
                         **step_stats(tp["ms"]), "tbps": tbps, "pct_of_peak": 100.0 * tbps * 1e3 / peak,
                         "bytes_per_step": int(tp["bytes_mean"]), **kr,
                         "traffic": recorded_traffic(kr["kernel"], workload_key(pc["w"], pc["mode"]))}
            del pc
            torch.cuda.empty_cache()
        out["per_config"] = per
    return out


def slowest_rank_ms(ms_local: float, world: int) -> float:
    """Step time of the whole job: the maximum of the ranks' mean step times."""
    if world == 1:
        return ms_local
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tbps(bytes_per_rank: float, ms_max: float, world: int) -> float:
    """Every rank decodes its own batch (replicas, weak scaling): total bytes over the slowest rank's time."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e12


def cpu_baseline(w, mode: str, budget_s: float = 12.0) -> dict:
    """The oracle as it stands, on all host cores, repeated on the full workload for ~budget_s."""
    import oracle
    import workloads as wl

    threads = oracle.hardware_threads()
    table = w.table
    if w.append_steps:
        table = wl.table_after_append(w.table)
    layout = "nhd" if mode == "contiguous_nhd" else "hnd"
    if mode.startswith("contiguous"):
        kc, vc, nv = wl.contiguous_copy(w)
        if layout == "nhd":
            kc, vc = np.ascontiguousarray(kc.transpose(0, 2, 1, 3)), np.ascontiguousarray(vc.transpose(0, 2, 1, 3))
    if mode == "paged_fp8":
        k8, v8, ks, vs = wl.fp8_pool(w)
    n, t0 = 0, time.perf_counter()
    while True:
        if mode.startswith("contiguous"):
            oracle.contiguous_decode(w.q, kc, vc, w.num_qo_heads, nv, w.sm_scale, w.dtype, threads, layout=layout)
        elif mode == "paged_fp8":
            t = w.table
            oracle.paged_decode_fp8(w.q, k8, v8, ks, vs, t.indices, t.indptr, t.last_page_len, w.num_qo_heads,
                                    w.num_kv_heads, w.head_dim, t.page_size, w.sm_scale, w.dtype, threads)
        else:
            oracle.paged_decode_workload(w, table=table, threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (n >= 1 and el * (n + 1) / n > 3 * budget_s):
            break
    per = el / n
    value = algorithmic_bytes(w, table, mode) / per / 1e12
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"full {w.name} decode, {n} call(s), {per * 1e3:.1f} ms per call on {threads} threads"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=["tiny", "llama3_8b", "llama3_8b_fp8", "long_context", "long_context_contiguous",
                             "long_context_nhd", "ragged_70b", "mha_append"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--append", default="fused", choices=["fused", "separate"],
                    help="append workloads: one fused append + decode launch, or an append launch then a decode")
    ap.add_argument("--fp8-kernel", default="mma", choices=["mma", "tcgen05"],
                    help="E4M3 pools: the mma.sync kernel (default) or the tcgen05 one where it applies")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the extra workloads timed after the headline one (one GPU only)")
    ap.add_argument("--quick", action="store_true",
                    help="decode steps only: no copy-peak, end-to-end or CPU-baseline legs (for profiler runs)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        w, mode = load_workload(args.config)
        for _ in range(args.warmup):
            pass  # the oracle has no warm state; warm-up calls would only repeat the timing
        cb = cpu_baseline(w, mode, budget_s=max(5.0, min(60.0, 2.0 * args.steps)))
        per_ms = algorithmic_bytes(w, mode=mode) / (cb["value"] * 1e12) * 1e3
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if mode == "paged_fp8" else w.dtype,
                "data": "synthetic",
                "config": {"workload": w.name}, "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    r = run_gpu(args, rank, world, local_rank)
    ms_max = slowest_rank_ms(r["ms_mean"], world)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    w = r["w"]
    tbps = whole_job_tbps(r["bytes_mean"], ms_max, world)
    peaks = measured_peaks()
    prof = r["prof"]
    kr = kernel_roofline({"w": w, "mode": r["mode"]}, {"prof": prof, "decode_bytes_mean": r["decode_bytes_mean"]},
                         peaks["hbm_gbs"])
    traffic = recorded_traffic(kr["kernel"], workload_key(w, r["mode"]))
    roofline = {"bound": "hbm", "achieved": kr["achieved"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": kr["frac"], "traffic": traffic, "peak_source": peaks["source"], "kernel": kr["kernel"],
                "kernel_us": kr["kernel_us"], "merge_us": kr["merge_us"], "append_us": kr["append_us"],
                "copy_kernel_gbs": r["copy_gbs"],
                "timing": "kernel events from a second pass over the same K steps"}
    cb = None if (args.no_cpu_baseline or args.quick) else cpu_baseline(w, r["mode"])
    # library kernels in the timed steps: decode + merge + append; the L2 flush is a torch fill
    launches = prof["decode_launches"] + prof["merge_launches"] + prof["append_launches"]
    ms = r["ms_all"]
    line = {
        "metric": METRIC, "value": tbps, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if r["mode"] == "paged_fp8" else w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "mode": r["mode"] + (f", append {args.append}" if w.append_steps else "")
                   + (", tcgen05 kernel" if r["mode"] == "paged_fp8" and args.fp8_kernel == "tcgen05" else ""),
                   "batch": w.batch, "num_qo_heads": w.num_qo_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "kv_tokens": int(w.table.kv_len().sum()), "bytes_per_step": int(r["bytes_mean"]),
                   "l2": "flushed before every timed step, outside the timed events: 512 MB written, then "
                         "256 MB read so the step starts with a cold, clean L2",
                   "parallelism": f"replicas x{world}",
                   "launch": f"the timed steps are queued behind a {PREROLL_S * 1e3:.0f} ms spin kernel, so the "
                             "host runs ahead of the GPU; garbage collection off while timing"},
        "us_per_call": ms_max * 1e3,
        **step_stats(ms),
        "us_steps": [round(x * 1e3, 2) for x in ms] if len(ms) <= 64 else None,
        "rows_per_s": world * w.batch / (ms_max * 1e-3),
        "pct_of_peak": 100.0 * tbps * 1e3 / world / peaks["hbm_gbs"],
        "roofline": roofline, "cpu_baseline": cb, "e2e": r["e2e"], "gpu_launches": launches,
        "clocks": r["clocks"],
    }
    if r["per_config"]:
        line["per_config"] = r["per_config"]
    print(json.dumps(line))
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
