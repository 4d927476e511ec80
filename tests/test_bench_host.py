"""Host-side logic of bench.py, on the CPU: the replica ranks' barrier and max-over-ranks timing
(world size 2 over gloo, as torchrun would launch it), and the useful-work counts that turn a
timing into TFLOP/s and GB/s, checked against the oracle's own counts."""
import os
import socket
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from oracle import sdpa_varlen_oracle as O  # noqa: E402
from workloads import synth  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, local = bench.dist_setup()
    bench.barrier(w)
    # each rank's "elapsed time": the job's time is the slowest rank's
    t = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    out.put((r, local, w, t))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_replica_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert [g[1] for g in got] == [0, 1]
    assert all(g[2] == 2 for g in got)
    assert all(g[3] == 2.5 for g in got)  # max over the two ranks, on both


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (1, 0, 0)
    assert bench.max_over_ranks(3.25, w) == 3.25


@pytest.mark.parametrize("index", [0, 1, 3, 4])
def test_useful_work_matches_the_oracle_counts(index):
    wl = synth.workload(index)
    for c in wl.calls:
        flops, kv, _ = bench.useful_work(c)
        assert flops == O.useful_flops(c.seq_info, c.T, c.Hq, c.D, c.causal, c.window, c.rows, c.cols)
        assert kv == O.useful_kv_bytes(c.seq_info, c.T, c.Hkv, c.D, c.window, c.rows, c.cols)


def test_useful_work_skips_invalid_and_overlapping_segments():
    rng = np.random.default_rng(5)
    c = synth.random_call(rng, D=64, Hq=4, Hkv=2, T=64, S=6, rows=256, cols=3, causal=True,
                          window=0, max_q=12, max_kv=200, gen_seed=2)
    seq = np.array(c.seq_info, copy=True)
    seq[0] = (0, 8, 0, 50)
    seq[1] = (4, 8, 1, 60)    # overlaps segment 0: both dropped
    seq[2] = (20, 4, 7, 30)   # column out of range: skipped
    c.seq_info = seq
    flops, kv, _ = bench.useful_work(c)
    assert flops == O.useful_flops(seq, c.T, c.Hq, c.D, c.causal, c.window, c.rows, c.cols)
    assert kv == O.useful_kv_bytes(seq, c.T, c.Hkv, c.D, c.window, c.rows, c.cols) - \
        sum(O.needed_span(int(s[1]), int(s[3]), c.window) * c.Hkv * c.D * 4 for s in seq[:2]
            if not O.segment_status(s, c.T, c.rows, c.cols, c.window))


def test_useful_work_of_the_one_store_mixed_step_uses_each_segments_mode():
    c = synth.workload(5).calls[0]
    flops, kv, _ = bench.useful_work(c)
    _, lo, hi, st = O.visible_interval(c.seq_info, c.T, True, 0, c.rows, c.cols, seg_mode=c.seg_mode)
    assert st == 0
    assert flops == 4 * c.D * c.Hq * int(np.maximum(hi - lo, 0).sum())
    assert kv == sum(O.needed_span(int(s[1]), int(s[3]), int(m[1])) * c.Hkv * c.D * 4
                     for s, m in zip(c.seq_info, c.seg_mode))
    # the same segments as two call-level calls (targets causal W=4096, drafts non-causal)
    t, d = c.seg_mode[:, 0] == 1, c.seg_mode[:, 0] == 0
    f_t = O.useful_flops(c.seq_info[t], c.T, c.Hq, c.D, True, 4096, c.rows, c.cols)
    f_d = O.useful_flops(c.seq_info[d], c.T, c.Hq, c.D, False, 0, c.rows, c.cols)
    assert flops == f_t + f_d


def test_reference_arm_prints_one_contract_line_on_the_cpu():
    import json
    import subprocess

    out = subprocess.run([sys.executable, os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"),
                          "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] >= 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert "cpu_model" in d["cpu_baseline"] and "blas_threads" in d["cpu_baseline"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_clock_window_takes_only_the_samples_inside_it():
    # (time, sm_mhz, max_mhz, reason bits, power W)
    samples = [(0.5, 900.0, 2070.0, 0x1, 100.0),        # before: idle, lower clock
               (1.0, 2070.0, 2070.0, 0x0, 800.0),
               (1.1, 2040.0, 2070.0, 0x4, 1390.0),      # power cap inside the window
               (1.2, 2070.0, 2070.0, 0x0, 900.0),
               (2.5, 1200.0, 2070.0, 0x40, 700.0)]      # after: thermal, outside the window
    w = bench.summarize_clocks(samples, 1.0, 1.2, "test")
    assert w["samples"] == 3 and w["sm_mhz"] == 2070.0 and w["sm_min_mhz"] == 2040.0
    assert w["sm_max_mhz"] == 2070.0 and w["reasons"] == ["sw_power_cap"] and w["power_w_max"] == 1390.0
    empty = bench.summarize_clocks(samples, 3.0, 4.0, "test")
    assert empty["samples"] == 0 and empty["sm_mhz"] is None and "note" in empty


def test_step_statistics_are_median_mean_and_deciles():
    ms = [1.0 + 0.1 * k for k in range(11)]  # 1.0 .. 2.0
    st = bench.percentiles(ms)
    assert st["median"] == pytest.approx(1.5) and st["mean"] == pytest.approx(1.5)
    assert st["p10"] == pytest.approx(1.1) and st["p90"] == pytest.approx(1.9) and st["n"] == 11


def test_stored_traffic_goes_null_when_the_kernel_source_changes(monkeypatch):
    name = next(iter(bench.NCU_TRAFFIC))
    nbytes, kind, sha = bench.NCU_TRAFFIC[name]
    monkeypatch.setitem(bench.NCU_TRAFFIC, name, (nbytes, kind, bench.kernel_sha(kind)))
    assert bench.ncu_traffic(name) == nbytes
    monkeypatch.setitem(bench.NCU_TRAFFIC, name, (nbytes, kind, "0" * 16))
    assert bench.ncu_traffic(name) is None
    assert bench.ncu_traffic("no such workload") is None


def test_every_per_config_workload_is_known_and_builds():
    for name in bench.PER_CONFIG:
        assert name in bench.WORKLOADS
    for name in ("prefill_d256", "ring_prefill"):
        wl = synth.workload(bench.WORKLOADS[name])
        flops, kv, _ = bench.useful_work(wl.calls[0])
        c = wl.calls[0]
        assert flops == O.useful_flops(c.seq_info, c.T, c.Hq, c.D, c.causal, c.window, c.rows, c.cols) > 0
