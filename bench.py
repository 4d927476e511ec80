"""Benchmark of length-aware GQA attention on one GB300 (replicas on N GPUs).

Prints one JSON line (rank 0).  A step is one pass of the whole path (scheduler, attention
kernels, combine) over one synthetic batch, inputs resident in HBM.  The workload defaults to
the long-context causal GQA prefill with D=128, Lq=4096, Lkv=131072, Hq=16, Hkv=2 (the
D=128 row of the operator table on "[CUDA] Use Triton TMA for long-context causal prefill").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

value: useful (mask-aware) TFLOP/s for prefill workloads, useful KV GB/s for decode-like
ones, whole job (all ranks).  The L2 is flushed (a 512 MiB write) between timed steps,
outside each step's events.  `roofline` reports the dominant kernel, timed with CUDA events
recorded by the library on the launch stream; `e2e` repeats the measurement through the C
interface from pinned host buffers (H2D of the step's inputs and D2H of its output inside
the timed region); `cpu_baseline` times the fp64 CPU oracle on a bounded sample.
"""

from __future__ import annotations

import argparse
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

WORKLOADS = {
    "tiny": 0, "prefill_d64": 1, "prefill_d128": 2, "decode": 3, "mixed": 4, "decode_append": 3,
    "seq_clone": -1, "mixed_modes": 5,
}
# seq_clone workload: one column of a [rows, cols, Hkv, D] store pair copied whole into another
CLONE_SHAPE = (32768, 9, 8, 128)
# workloads whose step first writes its new keys and values into the stores (sdpa_varlen_append)
APPEND = {"decode_append"}
PREFILL_LIKE = {"tiny", "prefill_d64", "prefill_d128"}
METRIC = "varlen GQA attention TFLOP/s (prefill) & KV GB/s (decode), % of roofline"
L2_FLUSH_BYTES = 512 << 20
# DRAM bytes (read + write) of the dominant kernel per step, from one ncu capture of the same
# bench line on a GB300 (dram__bytes_read.sum + dram__bytes_write.sum; the file under profiles/
# named for the kernel and workload gives the command).  They describe the kernel source they
# were taken on: a kernel change makes them stale until the capture is repeated.
NCU_TRAFFIC_BYTES = {
    "prefill_d128": 2304273152 + 37948416,  # sdpa_prefill_kernel<128>, one launch
    "prefill_d64": 9514752 + 0,             # sdpa_prefill_kernel<64>, one launch
    "decode": 141780224 + 3403008,          # sdpa_splitk_kernel<128>, one launch
    "mixed": 135080704 + 4520448 + 150389248 + 5599488,  # sdpa_splitk_kernel<128>, both calls
    "mixed_modes": 217293568 + 8046592,    # sdpa_splitk_kernel<128>, one launch
    "decode_append": 141788928 + 3189504,  # sdpa_splitk_kernel<128>, one launch
    # sdpa_clone_kernel: writes still dirty in L2 when the kernel ends are not counted
    "seq_clone": 134240768 + 84825600,
}


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


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


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
    el = max(el, 1e-9)
    value = done_flops / el / 1e12 if prefill_like else done_bytes / el / 1e9
    return {"value": value, "unit": "TFLOP/s" if prefill_like else "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the last {n_rows} packed rows (all heads) of {wl.name}: {el:.1f} s of fp64 NumPy "
                      f"on {cores} host cores (BLAS threads: default)"}


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
                         "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_clone(args, world, rank, local):
    """The column clone: K and V of one whole column (rows x Hkv x D) read once and written
    once per step, against the HBM copy roofline; the oracle's copy times the CPU leg."""
    import torch

    import varlen_gqa_attention_gb300 as pkg
    from oracle import sdpa_varlen_oracle as O

    rows, cols, Hkv, D = CLONE_SHAPE
    name = f"seq_clone_store{rows}x{cols}x{Hkv}x{D}_full_column"
    moved = 2 * 2 * rows * Hkv * D * 2  # K and V, read and written
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
        print(json.dumps({"impl": "reference", "metric": "seq_clone GB/s moved", "value": v, "unit": "GB/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "config": {"workload": name},
                          "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                           "sample": f"{n_cpu} rows of one column"},
                          "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    g = torch.Generator().manual_seed(args.seed)
    k = torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        pkg.sdpa_seq_clone(k, v, 0, cols - 1, rows)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e0.record()
        pkg.sdpa_seq_clone(k, v, i % (cols - 1), cols - 1, rows)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    barrier(world)
    clk = clocks.stop()
    mean = max_over_ranks(statistics.mean(ms), world)
    value = world * moved / (mean * 1e-3) / 1e9
    hbm, _, _, src = read_peaks()
    # end to end: the column pair goes up from pinned host memory, the clone runs, and the
    # destination column comes back
    hk, hv = k.cpu().pin_memory(), v.cpu().pin_memory()
    hcol = torch.empty((rows, Hkv, D), dtype=torch.bfloat16).pin_memory()
    e2e = []
    for i in range(max(2, args.steps // 2)):
        e0.record()
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        pkg.sdpa_seq_clone(k, v, 0, cols - 1, rows)
        hcol.copy_(k[:, cols - 1], non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        e2e.append(e0.elapsed_time(e1))
    e2e_ms = statistics.mean(e2e)
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n_cpu = 4096
        kc = torch.zeros((n_cpu, 2, Hkv, D), dtype=torch.bfloat16)
        t0 = time.perf_counter()
        O.seq_clone(kc, kc, 0, 1, n_cpu)
        el = time.perf_counter() - t0
        cpu = {"value": 2 * 2 * n_cpu * Hkv * D * 2 / el / 1e9, "unit": "GB/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle", "sample": f"{n_cpu} rows of one column ({el:.2f} s)"}
    print(json.dumps({
        "metric": "seq_clone GB/s moved", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "l2": "flushed between steps"},
        "roofline": {"bound": "hbm", "achieved": moved / (mean * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": moved / (mean * 1e-3) / 1e9 / hbm, "traffic": NCU_TRAFFIC_BYTES.get("seq_clone"), "kernel": "clone",
                     "peak_source": f"{src} HBM copy"},
        "e2e": {"value": moved / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": 2 * hk.numel() * 2,
                "d2h_bytes_per_step": hcol.numel() * 2, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps, "clocks": clk, "cpu_baseline": cpu,
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
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup()
    from workloads import synth

    if args.workload == "seq_clone":
        run_clone(args, world, rank, local)
        return
    wl = synth.workload(WORKLOADS[args.workload], seed=args.seed)
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
        return

    import torch

    import varlen_gqa_attention_gb300 as pkg

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    prefill_like = args.workload in PREFILL_LIKE

    # device-resident inputs, outputs and workspaces
    calls = []
    T_total = max(c.row_end or c.T for c in wl.calls)
    out = torch.empty((T_total, wl.calls[0].Hq, wl.calls[0].D), dtype=torch.bfloat16, device=dev)
    for c in wl.calls:
        d = dict(call=c, q=c.q.to(dev), k=c.k_store.to(dev), v=c.v_store.to(dev),
                 seq=torch.from_numpy(c.seq_info).to(dev),
                 ws=torch.empty(pkg.workspace_bytes(c.T, c.Hq, c.Hkv, c.D, len(c.seq_info)),
                                dtype=torch.uint8, device=dev))
        d["out"] = out[c.row_begin:(c.row_end or c.T)]
        if c.seg_mode is not None:
            d["md"] = torch.from_numpy(np.ascontiguousarray(c.seg_mode, dtype=np.int32)).to(dev)
        if args.workload in APPEND:
            g = torch.Generator().manual_seed(1000 + args.seed)
            shape = (c.T, c.Hkv, c.D)
            d["kn_host"] = torch.randn(shape, generator=g).to(torch.bfloat16)
            d["vn_host"] = torch.randn(shape, generator=g).to(torch.bfloat16)
            d["kn"], d["vn"] = d["kn_host"].to(dev), d["vn_host"].to(dev)
        calls.append(d)

    def attend(d):
        c = d["call"]
        if "kn" in d:
            pkg.sdpa_varlen_append(d["q"], d["kn"], d["vn"], d["k"], d["v"], d["seq"], causal=c.causal,
                                   window=c.window, scale=c.scale, out=d["out"], workspace=d["ws"])
        elif "md" in d:
            pkg.sdpa_varlen_modes(d["q"], d["k"], d["v"], d["seq"], d["md"], scale=c.scale, out=d["out"],
                                  workspace=d["ws"])
        else:
            pkg.sdpa_varlen(d["q"], d["k"], d["v"], d["seq"], causal=c.causal, window=c.window,
                            scale=c.scale, out=d["out"], workspace=d["ws"])
    flops = sum(useful_work(c)[0] for c in wl.calls)
    kv_bytes = sum(useful_work(c)[1] for c in wl.calls)
    qo_bytes = sum(useful_work(c)[2] for c in wl.calls)
    if args.workload in APPEND:
        # the step's new K and V rows, read once and written once (every covered row writes:
        # kv_end >= q_len in these workloads)
        kv_bytes += sum(useful_work(c)[2] // (4 * c.Hq * c.D) * c.Hkv * c.D * 2 * 2 * 2 for c in wl.calls)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        for i, d in enumerate(calls):
            if evs is not None:
                pkg.set_timing_events(evs[i])
            attend(d)
        if evs is not None:
            pkg.set_timing_events(None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The step is captured as CUDA graphs and replayed: no host submission gaps inside a step.
    # graph_s is the step as a caller runs it (the library chains its kernels with programmatic
    # dependent launch) and gives the timed value; graph_k has the library's timing events at
    # every kernel boundary (each kernel then runs alone) and gives the per-kernel times that
    # the roofline uses.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in calls]
    for e in (e for b in ev for e in b):
        e.record(stream)  # torch creates the CUDA event on its first record
    torch.cuda.synchronize()
    graph_k = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_k):
        step(ev)
    graph_s = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_s):
        step()
    for _ in range(args.warmup):
        graph_s.replay()
        graph_k.replay()
    torch.cuda.synchronize()
    e_beg = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    step_ms = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)  # L2 flush outside the step's events
        e_beg.record(stream)
        graph_s.replay()
        e_end.record(stream)
        torch.cuda.synchronize()
        step_ms.append(e_beg.elapsed_time(e_end))
    barrier(world)
    clk = clocks.stop()

    # per-kernel breakdown, same L2 flush, outside the timed steps
    times = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        graph_k.replay()
        torch.cuda.synchronize()
        times.append([[ev[i][a].elapsed_time(ev[i][a + 1]) for a in range(4)] for i in range(len(calls))])
    kern_ms = {"sched": [], "prefill": [], "splitk": [], "combine": []}
    for k in range(args.steps):
        for i in range(len(calls)):
            e = times[k][i]
            kern_ms["sched"].append(e[0])
            kern_ms["prefill"].append(e[1])
            kern_ms["splitk"].append(e[2])
            kern_ms["combine"].append(e[3])
    ms = statistics.mean(step_ms)
    ms_all = max_over_ranks(ms, world)
    if prefill_like:
        value = world * flops / (ms_all * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        value = world * kv_bytes / (ms_all * 1e-3) / 1e9
        unit = "GB/s"

    # dominant kernel and its roofline
    hbm, bf16, bf16_sus, peak_src = read_peaks()
    means = {k: statistics.mean(v) * len(calls) for k, v in kern_ms.items()}
    dom = max(("prefill", "splitk"), key=lambda k: means[k])
    dom_ms = means[dom]
    if prefill_like:
        achieved = flops / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                "frac": achieved / bf16, "traffic": NCU_TRAFFIC_BYTES.get(args.workload), "kernel": dom,
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    else:
        alg = kv_bytes + qo_bytes
        achieved = alg / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": NCU_TRAFFIC_BYTES.get(args.workload), "kernel": dom,
                "peak_source": f"{peak_src} HBM copy"}

    # end to end through the C interface from pinned host buffers
    host = []
    h2d = 0
    for d in calls:
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
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    d2h = hout.numel() * 2

    def e2e_step():
        for d, (hq, hk, hv, hs) in zip(calls, host):
            d["q"].copy_(hq, non_blocking=True)
            d["k"].copy_(hk, non_blocking=True)
            d["v"].copy_(hv, non_blocking=True)
            d["seq"].copy_(hs, non_blocking=True)
            if "kn" in d:
                d["kn"].copy_(d["kn_pin"], non_blocking=True)
                d["vn"].copy_(d["vn_pin"], non_blocking=True)
            if "md" in d:
                d["md"].copy_(d["md_pin"], non_blocking=True)
            attend(d)
        hout.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e = max_over_ranks(statistics.mean(e2e_ms), world)
    e2e_val = world * (flops if prefill_like else kv_bytes) / (e2e * 1e-3) / (1e12 if prefill_like else 1e9)

    # scheduler, split-K and combine per call, plus the prefill kernel when the head group
    # divides its 128-row tile, plus the KV append kernel on the append workload
    launches = args.steps * sum(3 + (1 if 128 % (d["call"].Hq // d["call"].Hkv) == 0 else 0) +
                                (1 if "kn" in d else 0) for d in calls)

    if rank != 0:
        return
    base = None
    if not args.no_cpu_baseline:
        base = cpu_baseline(wl, prefill_like)
    vs = None
    if args.workload == "prefill_d128":
        vs = value / 160.1  # RTX 5090 Triton TMA, 27.039 ms on this shape (pages' operator table)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_all, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + ("+kv_append" if args.workload in APPEND else ""),
                   "description": wl.description, "seed": args.seed,
                   "l2": "flushed between steps (512 MiB write outside the step's events)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "useful_tflop_per_step": flops / 1e12, "kv_gb_per_step": kv_bytes / 1e9},
        "roofline": roof,
        "kernel_ms": {k: statistics.mean(v) for k, v in kern_ms.items()},
        "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e},
        "gpu_launches": launches,
        "clocks": clk,
        "cpu_baseline": base,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
