"""Benchmark of length-aware GQA attention on one GB300 (replicas on N GPUs).

Prints one JSON line (rank 0).  A step is one pass of the whole path (scheduler, attention
kernels, combine) over one synthetic batch, inputs resident in HBM.  The headline workload is
the long-context causal GQA prefill with D=128, Lq=4096, Lkv=131072, Hq=16, Hkv=2 (the D=128
row of the operator table on "[CUDA] Use Triton TMA for long-context causal prefill"); the
line also carries a `per_config` block with every other workload, each timed and clocked on
its own.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                  [--no-per-config] [--no-cpu-baseline]

value: useful (mask-aware) TFLOP/s for prefill workloads, useful KV GB/s for decode-like
ones, whole job (all ranks).  Each step is a CUDA-graph replay; the L2 is flushed between
timed steps, outside each step's events, by reading a 512 MiB buffer (so the L2 holds none of
the step's inputs, and no dirty lines: a write flush leaves up to the L2's size of dirty lines
whose write-back would land in the next step's timed region); `ms_per_step` is the median step,
with the mean and the 10th / 90th percentiles beside it.  `roofline` reports the dominant
kernel, timed with CUDA events that the library records on the launch stream; `e2e` repeats
the measurement through the C interface from pinned host buffers (H2D of the step's inputs
and D2H of its output inside the timed region); `cpu_baseline` times the fp64 CPU oracle on
a bounded sample.  Clocks and throttle reasons are sampled from NVML every ~2 ms (nvidia-smi
every 100 ms where NVML cannot be loaded); each timed region reports the samples taken
inside it.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "tiny": 0, "prefill_d64": 1, "prefill_d128": 2, "decode": 3, "mixed": 4, "decode_append": 3,
    "seq_clone": -1, "mixed_modes": 5, "prefill_d256": 6, "ring_prefill": 7,
}
# the default line's per-config block, in this order (the headline workload first)
PER_CONFIG = ["prefill_d128", "tiny", "prefill_d64", "prefill_d256", "ring_prefill", "decode",
              "decode_append", "mixed", "mixed_modes", "seq_clone"]
# seq_clone workload: one column of a [rows, cols, Hkv, D] store pair copied whole into another
CLONE_SHAPE = (32768, 9, 8, 128)
# workloads whose step first writes its new keys and values into the stores (sdpa_varlen_append)
APPEND = {"decode_append"}
PREFILL_LIKE = {"tiny", "prefill_d64", "prefill_d128", "prefill_d256", "ring_prefill"}
METRIC = "varlen GQA attention TFLOP/s (prefill) & KV GB/s (decode), % of roofline"
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evicts the L2 by reading a buffer four times its size (clean lines only: nothing of the
    next step's inputs stays cached and nothing dirty is left to write back)."""

    def __init__(self, dev):
        import torch

        self.buf = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def fill_(self, k):
        self.sink.add_(self.buf.sum())
CSRC = os.path.join(ROOT, "varlen_gqa_attention_gb300", "csrc")
# the sources each kernel is built from (their hash ties a traffic figure to the code it was
# measured on)
KERNEL_SOURCES = {
    # the scheduler decides what the attention kernels read and write (pieces, partial slots)
    "prefill": ["prefill.cu", "prefill_pair.cu", "tc.cuh", "common.cuh", "sched.cu"],
    "splitk": ["splitk.cu", "common.cuh", "sched.cu"],
    "clone": ["append.cu", "common.cuh"],
}
# DRAM bytes (read + write) of the dominant kernel per step, from one ncu capture of the same
# bench line on a GB300 (dram__bytes_read.sum + dram__bytes_write.sum; the file under profiles/
# named for the kernel and workload gives the command), with the hash of that kernel's sources
# when it was taken.  A kernel whose sources hash differently now reports traffic null until
# the capture is repeated.
NCU_TRAFFIC = {
    "prefill_d128": (1207549440 + 65541888, "prefill", "91780631a32d4b44"),  # sdpa_prefill_pair_kernel<128>
    "prefill_d64": (9903616 + 512, "prefill", "91780631a32d4b44"),  # sdpa_prefill_pair_kernel<64>
    "prefill_d256": (334566912 + 47162368, "prefill", "91780631a32d4b44"),  # sdpa_prefill_kernel<256>
    "ring_prefill": (14966016 + 0, "prefill", "91780631a32d4b44"),  # sdpa_prefill_pair_kernel<128>
    "tiny": (159744 + 0, "splitk", "e448effc74ee4957"),  # sdpa_splitk_kernel<64> (tiny calls take the split-K route)
    "decode": (141723648 + 3188224, "splitk", "e448effc74ee4957"),  # sdpa_splitk_kernel<128>
    "decode_append": (141728000 + 3187456, "splitk", "e448effc74ee4957"),
    "mixed": (285199872 + 11369472, "splitk", "e448effc74ee4957"),  # both calls
    "mixed_modes": (220047104 + 8420096, "splitk", "e448effc74ee4957"),
    # sdpa_clone_kernel: writes still dirty in L2 when the kernel ends are not counted
    "seq_clone": (134241280 + 84925696, "clone", "c9b82a90a0e5fff4"),
}


def kernel_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """The stored DRAM traffic of the workload's dominant kernel, or None when there is none
    or the kernel's sources changed since it was captured."""
    t = NCU_TRAFFIC.get(workload)
    if t is None:
        return None
    nbytes, kind, sha = t
    return nbytes if kernel_sha(kind) == sha else None


def useful_work(call):
    """(flops, kv_bytes, q_out_bytes) the call must do: 4*D*Hq per (row, visible key) pair,
    K and V bytes of the union of each valid segment's visible positions, and q/out bytes of
    the rows valid segments cover."""
    T, rows, cols = call.T, call.rows, call.cols
    segs = np.asarray(call.seq_info, dtype=np.int64)
    if call.seg_mode is None:
        modes = [(bool(call.causal), int(call.window))] * len(segs)
    else:
        modes = [(bool(c), int(w)) for c, w in np.asarray(call.seg_mode, dtype=np.int64)]
    pairs = 0
    kv = 0
    covered = 0
    owners = np.zeros(T, dtype=np.int64)
    ok = []
    for (qs, ql, col, ke), (_, W) in zip(segs, modes):
        bad = ql < 0 or qs < 0 or qs + ql > T or col < 0 or col >= cols or ke < 0
        if not bad and ql > 0 and ke > 0:
            span = min(ke, ql + W - 1) if W > 0 else ke
            bad = span > rows
        ok.append(not bad)
        if not bad and ql > 0:
            owners[qs:qs + ql] += 1
    for (qs, ql, col, ke), good, (causal, W) in zip(segs, ok, modes):
        if not good or ql <= 0 or (owners[qs:qs + ql] > 1).any():
            continue
        p = ke - ql + np.arange(ql)
        hi = np.minimum(p + 1, ke) if causal else np.full(ql, ke)
        lo = np.maximum(0, p - W + 1) if W > 0 else np.zeros(ql, dtype=np.int64)
        pairs += int(np.maximum(hi - lo, 0).sum())
        if ke > 0:
            span = min(ke, ql + W - 1) if W > 0 else ke
            kv += span * call.Hkv * call.D * 2 * 2
        covered += ql
    return 4 * call.D * call.Hq * pairs, kv, 2 * covered * call.Hq * call.D * 2


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def percentiles(ms):
    """median, mean, 10th and 90th percentile of a list of step times."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "mean": float(a.mean()), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------

REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def summarize_clocks(samples, t0: float, t1: float, source: str):
    """Median SM clock, max clock and every throttle reason seen in the samples taken in
    [t0, t1].  A sample is (time, sm_mhz, max_mhz, reason_bits, power_w)."""
    win = [s for s in samples if t0 <= s[0] <= t1]
    if not win:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": source,
                "note": "no clock sample fell inside the timed region"}
    sm = [s[1] for s in win]
    reasons = sorted({name for s in win for bit, name in REASON_BITS.items() if s[3] & bit})
    pw = [s[4] for s in win if s[4] is not None]
    return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(s[2] for s in win),
            "reasons": reasons, "samples": len(win), "source": source,
            "power_w_max": max(pw) if pw else None}


class ClockSampler:
    """SM clock, maximum clock, power and throttle reasons of one GPU, sampled in a background
    thread: from NVML (libnvidia-ml through ctypes) every ~2 ms, else from `nvidia-smi -lms
    100`.  Only reads; sets nothing.  Each sample carries the host time it was taken, so that
    every timed region reports the samples inside it (`window`)."""

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.cuda_index = cuda_index
        self.period = period_s
        self.samples = []
        self.source = "none"
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _nvml_handle(self):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        bus = None
        try:
            import torch

            p = torch.cuda.get_device_properties(self.cuda_index)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except Exception:  # noqa: BLE001 - fall back to the index
            bus = None
        rc = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) if bus else 1
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _nvml_loop(self, lib, h, reasons_fn):
        clk, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.monotonic()
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                r = reasons_fn(h, ctypes.byref(rs))
                p = lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
                self.samples.append((t, float(clk.value), float(mx.value), int(rs.value) if r == 0 else 0,
                                     pw.value / 1000.0 if p == 0 else None))
            time.sleep(self.period)

    def _smi_loop(self):
        for line in self._proc.stdout:
            t = time.monotonic()
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                pw = float(parts[2])
            except ValueError:
                pw = None
            bits = 0
            for bit, val in zip((0x8, 0x40, 0x20, 0x4), parts[3:7]):
                if val.lower().startswith("active"):
                    bits |= bit
            self.samples.append((t, sm, mx, bits, pw))

    def start(self):
        try:
            lib, h, rf = self._nvml_handle()
            self.source = f"nvml every {self.period * 1e3:.0f} ms"
            self._thread = threading.Thread(target=self._nvml_loop, args=(lib, h, rf), daemon=True)
            self._thread.start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.cuda_index), f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi every 100 ms"
            self._thread = threading.Thread(target=self._smi_loop, daemon=True)
            self._thread.start()
        except (OSError, FileNotFoundError):
            self.source = "unavailable"

    def window(self, t0: float, t1: float):
        return summarize_clocks(list(self.samples), t0, t1, self.source)

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)


# ------------------------------------------------------------------------------------------
# ranks
# ------------------------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# the CPU oracle as a baseline
# ------------------------------------------------------------------------------------------

def cpu_info():
    """CPU model and the BLAS thread count the oracle's NumPy runs with."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
        if model is None:
            vend = [ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Vendor ID:")]
            model = vend[0] if vend else None
    except (OSError, subprocess.SubprocessError):
        pass
    blas = None
    try:
        for ln in open("/proc/self/maps"):
            path = ln.split()[-1]
            if "openblas" in path.lower() and ".so" in path:
                lib = ctypes.CDLL(path)
                for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                             "openblas_get_num_threads"):
                    f = getattr(lib, name, None)
                    if f is not None:
                        blas = int(f())
                        break
                if blas is not None:
                    break
    except OSError:
        pass
    return model, blas


def cpu_baseline(wl, prefill_like: bool, budget_s: float = 12.0):
    """Time the fp64 oracle, as it stands, on a bounded sample: the last packed rows of each
    call (the heaviest ones under causal masking).  A first call on 8 rows calibrates how
    many rows fit the time budget; the second call on that many rows is the sample."""
    from oracle import sdpa_varlen_oracle as O

    el = 0.0
    done_flops = 0
    done_bytes = 0
    n_rows = 0
    per_call = budget_s / len(wl.calls)
    for c in wl.calls:
        seg_id, lo, hi, _ = O.visible_interval(c.seq_info, c.T, c.causal, c.window, c.rows, c.cols,
                                               seg_mode=c.seg_mode)
        live = [t for t in range(c.T) if seg_id[t] >= 0]
        if not live:
            continue
        t0 = time.perf_counter()
        O.sdpa_varlen(c.q, c.k_store, c.v_store, c.seq_info, c.causal, c.window, c.scale,
                      rows_subset=live[-8:], seg_mode=c.seg_mode)
        cal = max(time.perf_counter() - t0, 1e-3)
        n = int(min(len(live), max(8, 8 * per_call / cal)))
        rows = live[-n:]
        t0 = time.perf_counter()
        O.sdpa_varlen(c.q, c.k_store, c.v_store, c.seq_info, c.causal, c.window, c.scale, rows_subset=rows,
                      seg_mode=c.seg_mode)
        el += time.perf_counter() - t0
        n_rows += len(rows)
        done_flops += 4 * c.D * c.Hq * int(np.maximum(hi[rows] - lo[rows], 0).sum())
        for s in sorted(set(int(seg_id[t]) for t in rows)):
            qs, ql, col, ke = (int(x) for x in c.seq_info[s])
            w = c.window if c.seg_mode is None else int(c.seg_mode[s][1])
            done_bytes += O.needed_span(ql, ke, w) * c.Hkv * c.D * 2 * 2
    cores = len(os.sched_getaffinity(0))
    model, blas = cpu_info()
    el = max(el, 1e-9)
    value = done_flops / el / 1e12 if prefill_like else done_bytes / el / 1e9
    return {"value": value, "unit": "TFLOP/s" if prefill_like else "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": model, "blas_threads": blas,
            "sample": f"the last {n_rows} packed rows (all heads) of {wl.name}: {el:.1f} s of fp64 NumPy "
                      f"on {cores} host cores ({model or 'cpu model unknown'}; BLAS threads: "
                      f"{blas if blas is not None else 'unknown'})"}


def run_reference(args, wl, world, rank):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample per step."""
    if rank != 0:
        return
    prefill_like = args.workload in PREFILL_LIKE
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(wl, prefill_like, budget_s=per_step)
    t0 = time.perf_counter()
    vals = [cpu_baseline(wl, prefill_like, budget_s=per_step) for _ in range(args.steps)]
    el = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    unit = vals[0]["unit"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "description": wl.description},
        "cpu_baseline": {"value": v, "unit": unit, "cores": vals[0]["cores"], "kind": "oracle",
                         "cpu_model": vals[0]["cpu_model"], "blas_threads": vals[0]["blas_threads"],
                         "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# GPU timing
# ------------------------------------------------------------------------------------------

def time_replays(replay, n: int, flush, stream):
    """n steps, each a call of `replay` bracketed by CUDA events on `stream`, the L2 flushed
    before each step outside its events; one synchronisation at the end.  Returns the step
    times (ms) and the host-time window the GPU work fell in."""
    import torch

    beg = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    end = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    t0 = time.monotonic()
    for k in range(n):
        flush.fill_(k & 0xFF)
        beg[k].record(stream)
        replay()
        end[k].record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    return [b.elapsed_time(e) for b, e in zip(beg, end)], t0, t1


class Prepared:
    """Device-resident inputs of one workload and the step that runs it through the binding."""

    def __init__(self, name, seed, dev):
        import torch

        import varlen_gqa_attention_gb300 as pkg
        from workloads import synth

        self.name = name
        self.pkg = pkg
        self.wl = synth.workload(WORKLOADS[name], seed=seed)
        wl = self.wl
        self.prefill_like = name in PREFILL_LIKE
        self.calls = []
        T_total = max(c.row_end or c.T for c in wl.calls)
        self.out = torch.empty((T_total, wl.calls[0].Hq, wl.calls[0].D), dtype=torch.bfloat16, device=dev)
        for c in wl.calls:
            d = dict(call=c, q=c.q.to(dev), k=c.k_store.to(dev), v=c.v_store.to(dev),
                     seq=torch.from_numpy(c.seq_info).to(dev),
                     ws=torch.empty(pkg.workspace_bytes(c.T, c.Hq, c.Hkv, c.D, len(c.seq_info)),
                                    dtype=torch.uint8, device=dev))
            d["out"] = self.out[c.row_begin:(c.row_end or c.T)]
            if c.seg_mode is not None:
                d["md"] = torch.from_numpy(np.ascontiguousarray(c.seg_mode, dtype=np.int32)).to(dev)
            if name in APPEND:
                g = torch.Generator().manual_seed(1000 + seed)
                shape = (c.T, c.Hkv, c.D)
                d["kn_host"] = torch.randn(shape, generator=g).to(torch.bfloat16)
                d["vn_host"] = torch.randn(shape, generator=g).to(torch.bfloat16)
                d["kn"], d["vn"] = d["kn_host"].to(dev), d["vn_host"].to(dev)
            self.calls.append(d)
        works = [useful_work(c) for c in wl.calls]
        self.flops = sum(w[0] for w in works)
        self.kv_bytes = sum(w[1] for w in works)
        self.qo_bytes = sum(w[2] for w in works)
        if name in APPEND:
            # the step's new K and V rows, read once and written once (every covered row writes:
            # kv_end >= q_len in these workloads)
            self.kv_bytes += sum(w[2] // (4 * c.Hq * c.D) * c.Hkv * c.D * 2 * 2 * 2 for w, c in zip(works, wl.calls))
        # scheduler, split-K and combine per call, plus the prefill kernel when the head group
        # divides its 128-row tile, the call's packed rows can fill one and the call can hold
        # the prefill route's minimum work (packed rows * Hkv * D * longest key span >= 2^30),
        # plus the KV append kernel on the append workload
        def pf(c):
            g = c.Hq // c.Hkv
            span = c.rows if (c.seg_mode is not None or c.window <= 0) else min(c.rows, c.T + c.window - 1)
            return 1 if 128 % g == 0 and c.T * g >= 128 and c.T * g * c.Hkv * c.D * span >= 2 ** 30 else 0
        self.launches_per_step = sum(3 + pf(d["call"]) + (1 if "kn" in d else 0) for d in self.calls)

    def attend(self, d):
        pkg, c = self.pkg, d["call"]
        if "kn" in d:
            pkg.sdpa_varlen_append(d["q"], d["kn"], d["vn"], d["k"], d["v"], d["seq"], causal=c.causal,
                                   window=c.window, scale=c.scale, out=d["out"], workspace=d["ws"])
        elif "md" in d:
            pkg.sdpa_varlen_modes(d["q"], d["k"], d["v"], d["seq"], d["md"], scale=c.scale, out=d["out"],
                                  workspace=d["ws"])
        else:
            pkg.sdpa_varlen(d["q"], d["k"], d["v"], d["seq"], causal=c.causal, window=c.window,
                            scale=c.scale, out=d["out"], workspace=d["ws"])

    def step(self, evs=None):
        for i, d in enumerate(self.calls):
            if evs is not None:
                self.pkg.set_timing_events(evs[i])
            self.attend(d)
        if evs is not None:
            self.pkg.set_timing_events(None)


def measure(prep: Prepared, steps: int, warmup: int, flush, clocks, world, min_timed_s: float = 0.0):
    """Times one workload: `steps` CUDA-graph replays of the step as a caller runs it (more
    when `min_timed_s` asks for a longer timed region, so that it holds clock samples), each
    followed, inside the same timed region, by a replay of a graph with the library's timing
    events at every kernel boundary (each kernel then runs alone) for the per-kernel times, so
    that both see the same clocks.  The L2 is flushed before every replay, outside the events.
    Returns the config block (value, step-time statistics, roofline, kernel times, clocks)."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        prep.step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in prep.calls]
    for e in (e for b in ev for e in b):
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize()
    graph_k = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_k):
        prep.step(ev)
    graph_s = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_s):
        prep.step()
    t0 = time.monotonic()
    for _ in range(warmup):
        graph_s.replay()
        graph_k.replay()
    torch.cuda.synchronize()
    est = max((time.monotonic() - t0) / max(1, warmup), 1e-5)
    n = steps
    if min_timed_s > 0:
        n = max(steps, min(20000, int(math.ceil(min_timed_s / (est + 4e-4)))))
    kern = {"sched": [], "prefill": [], "splitk": [], "combine": []}
    e_beg = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    step_ms = []
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.monotonic()
    for k in range(n):
        flush.fill_(k & 0xFF)
        e_beg.record(stream)
        graph_s.replay()
        e_end.record(stream)
        flush.fill_(k & 0xFF)
        graph_k.replay()
        torch.cuda.synchronize()
        step_ms.append(e_beg.elapsed_time(e_end))
        for i in range(len(prep.calls)):
            e = [ev[i][a].elapsed_time(ev[i][a + 1]) for a in range(4)]
            for key, val in zip(("sched", "prefill", "splitk", "combine"), e):
                kern[key].append(val)
    w1 = time.monotonic()
    barrier(world)
    clk = clocks.window(w0, w1)
    stats = percentiles(step_ms)
    med = max_over_ranks(stats["median"], world)
    if prep.prefill_like:
        value = world * prep.flops / (med * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        value = world * prep.kv_bytes / (med * 1e-3) / 1e9
        unit = "GB/s"
    hbm, bf16, _, peak_src = read_peaks()
    # per step: the median kernel time times the calls of a step
    kmed = {k: statistics.median(v) * len(prep.calls) for k, v in kern.items()}
    dom = max(("prefill", "splitk"), key=lambda k: kmed[k])
    dom_ms = kmed[dom]
    if prep.prefill_like:
        achieved = prep.flops / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                "frac": achieved / bf16, "traffic": ncu_traffic(prep.name), "kernel": dom,
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    else:
        alg = prep.kv_bytes + prep.qo_bytes
        achieved = alg / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": ncu_traffic(prep.name), "kernel": dom,
                "peak_source": f"{peak_src} HBM copy"}
    return {
        "workload": prep.wl.name + ("+kv_append" if prep.name in APPEND else ""),
        "value": value, "unit": unit, "steps": n, "ms_per_step": med,
        "ms": {"median": stats["median"], "mean": stats["mean"], "p10": stats["p10"], "p90": stats["p90"]},
        "roofline": roof,
        "kernel_ms": {k: v / len(prep.calls) for k, v in kmed.items()},  # median per call
        "gpu_launches": 2 * n * prep.launches_per_step,  # the step and its timed-kernels copy
        "clocks": clk,
        "useful_tflop_per_step": prep.flops / 1e12, "kv_gb_per_step": prep.kv_bytes / 1e9,
    }


def measure_e2e(prep: Prepared, steps: int, flush, world):
    """The same step through the public API from pinned host buffers: H2D of the step's inputs
    and D2H of its output inside the timed region."""
    import torch

    stream = torch.cuda.current_stream()
    host = []
    h2d = 0
    for d in prep.calls:
        c = d["call"]
        hq, hk, hv = c.q.pin_memory(), c.k_store.pin_memory(), c.v_store.pin_memory()
        hs = torch.from_numpy(c.seq_info.copy()).pin_memory()
        host.append((hq, hk, hv, hs))
        h2d += hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2 + hs.numel() * 4
        if "kn" in d:
            d["kn_pin"], d["vn_pin"] = d["kn_host"].pin_memory(), d["vn_host"].pin_memory()
            h2d += (d["kn_pin"].numel() + d["vn_pin"].numel()) * 2
        if "md" in d:
            d["md_pin"] = d["md"].cpu().pin_memory()
            h2d += d["md_pin"].numel() * 4
    hout = torch.empty(prep.out.shape, dtype=torch.bfloat16).pin_memory()
    d2h = hout.numel() * 2

    def e2e_step():
        for d, (hq, hk, hv, hs) in zip(prep.calls, host):
            d["q"].copy_(hq, non_blocking=True)
            d["k"].copy_(hk, non_blocking=True)
            d["v"].copy_(hv, non_blocking=True)
            d["seq"].copy_(hs, non_blocking=True)
            if "kn" in d:
                d["kn"].copy_(d["kn_pin"], non_blocking=True)
                d["vn"].copy_(d["vn_pin"], non_blocking=True)
            if "md" in d:
                d["md"].copy_(d["md_pin"], non_blocking=True)
            prep.attend(d)
        hout.copy_(prep.out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    ms, _, _ = time_replays(e2e_step, steps, flush, stream)
    med = max_over_ranks(statistics.median(ms), world)
    denom = (1e12 if prep.prefill_like else 1e9)
    work = prep.flops if prep.prefill_like else prep.kv_bytes
    return {"value": world * work / (med * 1e-3) / denom, "unit": "TFLOP/s" if prep.prefill_like else "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": med}


def measure_clone(args, dev, flush, clocks, world, min_timed_s: float = 0.0):
    """The column clone: K and V of one whole column (rows x Hkv x D) read once and written
    once per step, against the HBM copy roofline."""
    import torch

    import varlen_gqa_attention_gb300 as pkg

    rows, cols, Hkv, D = CLONE_SHAPE
    moved = 2 * 2 * rows * Hkv * D * 2  # K and V, read and written
    g = torch.Generator().manual_seed(args.seed)
    k = torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    for _ in range(args.warmup):
        pkg.sdpa_seq_clone(k, v, 0, cols - 1, rows)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    n = args.steps
    if min_timed_s > 0:
        n = max(n, int(math.ceil(min_timed_s / 2.5e-4)))
    it = iter(range(10 ** 9))
    barrier(world)
    ms, w0, w1 = time_replays(lambda: pkg.sdpa_seq_clone(k, v, next(it) % (cols - 1), cols - 1, rows), n,
                              flush, stream)
    barrier(world)
    stats = percentiles(ms)
    med = max_over_ranks(stats["median"], world)
    hbm, _, _, src = read_peaks()
    achieved = moved / (med * 1e-3) / 1e9
    block = {
        "workload": f"seq_clone_store{rows}x{cols}x{Hkv}x{D}_full_column",
        "value": world * achieved, "unit": "GB/s", "steps": n, "ms_per_step": med,
        "ms": {"median": stats["median"], "mean": stats["mean"], "p10": stats["p10"], "p90": stats["p90"]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": ncu_traffic("seq_clone"), "kernel": "clone", "peak_source": f"{src} HBM copy"},
        "gpu_launches": n, "clocks": clocks.window(w0, w1),
    }
    return block, (k, v, moved)


def run_clone(args, world, rank, local):
    """`--workload seq_clone`: the clone as the headline; the oracle's copy times the CPU leg."""
    import torch

    import varlen_gqa_attention_gb300 as pkg
    from oracle import sdpa_varlen_oracle as O

    rows, cols, Hkv, D = CLONE_SHAPE
    name = f"seq_clone_store{rows}x{cols}x{Hkv}x{D}_full_column"
    if args.impl == "reference":
        if rank != 0:
            return
        n_cpu = 4096
        k0 = torch.zeros((n_cpu, 2, Hkv, D), dtype=torch.bfloat16)
        t0 = time.perf_counter()
        for _ in range(args.warmup + args.steps):
            O.seq_clone(k0, k0, 0, 1, n_cpu)
        el = (time.perf_counter() - t0) / (args.warmup + args.steps)
        v = 2 * 2 * n_cpu * Hkv * D * 2 / el / 1e9
        cores = len(os.sched_getaffinity(0))
        model, blas = cpu_info()
        print(json.dumps({"impl": "reference", "metric": "seq_clone GB/s moved", "value": v, "unit": "GB/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "config": {"workload": name},
                          "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                           "cpu_model": model, "blas_threads": blas,
                                           "sample": f"{n_cpu} rows of one column"},
                          "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    clocks = ClockSampler(local)
    clocks.start()
    block, (k, v, moved) = measure_clone(args, dev, flush, clocks, world)
    # end to end: the column pair goes up from pinned host memory, the clone runs, and the
    # destination column comes back
    hk, hv = k.cpu().pin_memory(), v.cpu().pin_memory()
    hcol = torch.empty((rows, Hkv, D), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        pkg.sdpa_seq_clone(k, v, 0, cols - 1, rows)
        hcol.copy_(k[:, cols - 1], non_blocking=True)

    e2e_step()
    ms, _, _ = time_replays(e2e_step, max(2, args.steps // 2), flush, torch.cuda.current_stream())
    e2e_ms = max_over_ranks(statistics.median(ms), world)
    clocks.stop()
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n_cpu = 4096
        kc = torch.zeros((n_cpu, 2, Hkv, D), dtype=torch.bfloat16)
        t0 = time.perf_counter()
        O.seq_clone(kc, kc, 0, 1, n_cpu)
        el = time.perf_counter() - t0
        model, blas = cpu_info()
        cpu = {"value": 2 * 2 * n_cpu * Hkv * D * 2 / el / 1e9, "unit": "GB/s",
               "cores": len(os.sched_getaffinity(0)), "kind": "oracle", "cpu_model": model, "blas_threads": blas,
               "sample": f"{n_cpu} rows of one column ({el:.2f} s)"}
    print(json.dumps({
        "metric": "seq_clone GB/s moved", "value": block["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": block["ms_per_step"], "ms": block["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "l2": "flushed between steps (512 MiB read)"},
        "roofline": block["roofline"],
        "e2e": {"value": world * moved / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": 2 * hk.numel() * 2, "d2h_bytes_per_step": hcol.numel() * 2,
                "ms_per_step": e2e_ms},
        "gpu_launches": block["gpu_launches"], "clocks": block["clocks"], "cpu_baseline": cpu,
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="prefill_d128", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload (default: also every other workload)")
    ap.add_argument("--min-config-s", type=float, default=0.25,
                    help="shortest timed region of a per-config block, in seconds (clock samples)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup()
    from workloads import synth

    if args.workload == "seq_clone":
        run_clone(args, world, rank, local)
        return
    if args.impl == "reference":
        run_reference(args, synth.workload(WORKLOADS[args.workload], seed=args.seed), world, rank)
        return

    import torch

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    clocks = ClockSampler(local)
    clocks.start()
    try:
        prep = Prepared(args.workload, args.seed, dev)
        head = measure(prep, args.steps, args.warmup, flush, clocks, world)
        e2e = measure_e2e(prep, args.steps, flush, world)
        per_config = None
        if not args.no_per_config and args.workload == "prefill_d128":
            per_config = {"prefill_d128": {k: head[k] for k in ("workload", "value", "unit", "steps", "ms_per_step",
                                                                "ms", "roofline", "kernel_ms", "clocks")}}
            del prep
            torch.cuda.empty_cache()
            for name in PER_CONFIG[1:]:
                if name == "seq_clone":
                    block, _ = measure_clone(args, dev, flush, clocks, world, args.min_config_s)
                else:
                    p = Prepared(name, args.seed, dev)
                    block = measure(p, args.steps, args.warmup, flush, clocks, world, args.min_config_s)
                    del p
                torch.cuda.empty_cache()
                block.pop("useful_tflop_per_step", None)
                block.pop("kv_gb_per_step", None)
                per_config[name] = block
    finally:
        clocks.stop()

    if rank != 0:
        return
    wl = synth.workload(WORKLOADS[args.workload], seed=args.seed)
    base = None
    if not args.no_cpu_baseline:
        base = cpu_baseline(wl, args.workload in PREFILL_LIKE)
    vs = None
    if args.workload == "prefill_d128":
        vs = head["value"] / 160.1  # RTX 5090 Triton TMA, 27.039 ms on this shape (pages' operator table)
    # kernels of this library launched in the headline's timed region (each per-config block
    # counts its own)
    launches = head["gpu_launches"]
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "ms": head["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": vs, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": head["workload"], "description": wl.description, "seed": args.seed,
                   "l2": "flushed between steps by a 512 MiB read outside the step's events",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "useful_tflop_per_step": head["useful_tflop_per_step"], "kv_gb_per_step": head["kv_gb_per_step"]},
        "roofline": head["roofline"],
        "kernel_ms": head["kernel_ms"],
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": head["clocks"],
        "cpu_baseline": base,
    }
    if per_config:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
