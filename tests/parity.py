"""Helpers shared by the GPU parity tests: run a synthetic call through the CUDA library and
compare it with the CPU oracle.

Tolerance (bf16 outputs of fp32-accumulated attention on N(0,1) inputs, compared with the
fp64 oracle): max |err| <= 2e-2 and mean |err| <= 2e-3 over covered rows that see at least
one key; uncovered rows and rows that see no key must be exactly 0.
"""

from __future__ import annotations

import numpy as np
import torch

import varlen_gqa_attention_gb300 as pkg
from oracle import sdpa_varlen_oracle as O

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def run_call(call, dev, *, out=None, q=None, k=None, v=None, status=None, seq_override=None):
    q = call.q.to(dev) if q is None else q
    k = call.k_store.to(dev) if k is None else k
    v = call.v_store.to(dev) if v is None else v
    si = call.seq_info if seq_override is None else seq_override
    seq = torch.from_numpy(np.ascontiguousarray(si, dtype=np.int32)).to(dev)
    # a workspace full of 0xFF bytes (NaN floats, -1 ints): nothing may rely on its contents
    ws = torch.full((pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(si)),), 255,
                    dtype=torch.uint8, device=dev)
    return pkg.sdpa_varlen(q, k, v, seq, causal=call.causal, window=call.window, scale=call.scale,
                           out=out, status=status, workspace=ws)


def oracle(call, rows_subset=None, seq_override=None, k=None, v=None):
    si = call.seq_info if seq_override is None else seq_override
    return O.sdpa_varlen(call.q, call.k_store if k is None else k, call.v_store if v is None else v,
                         si, call.causal, call.window, call.scale, rows_subset=rows_subset)


def assert_matches(got: torch.Tensor, ref: np.ndarray, seg_id: np.ndarray, lo: np.ndarray,
                   hi: np.ndarray, rows=None, tag=""):
    g = got.double().cpu().numpy()
    rows = np.arange(g.shape[0]) if rows is None else np.asarray(rows)
    live = rows[(seg_id[rows] >= 0) & (hi[rows] > lo[rows])]
    empty = rows[(seg_id[rows] == O.UNCOVERED) | ((seg_id[rows] >= 0) & (hi[rows] <= lo[rows]))]
    if len(live):
        err = np.abs(g[live] - ref[live])
        assert np.isfinite(g[live]).all(), f"{tag}: non-finite output"
        assert err.max() <= MAX_ABS, f"{tag}: max abs err {err.max():.4g}"
        assert err.mean() <= MEAN_ABS, f"{tag}: mean abs err {err.mean():.4g}"
    if len(empty):
        bits = got[torch.as_tensor(empty, device=got.device)].view(torch.int16)
        assert bool((bits == 0).all()), f"{tag}: uncovered/empty rows are not exactly 0"
    return (np.abs(g[live] - ref[live]).max() if len(live) else 0.0)


def check_call(call, dev, rows_subset=None, tag=""):
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = run_call(call, dev, status=status)
    torch.cuda.synchronize()
    ref, seg_id, st = oracle(call, rows_subset=rows_subset)
    _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, call.causal, call.window, call.rows, call.cols)
    assert int(status.item()) == st, f"{tag}: status {int(status.item())} != {st}"
    return assert_matches(got, ref, seg_id, lo, hi, rows=rows_subset, tag=tag)


def poison_invisible(call, value=float("nan")):
    """Copies of the stores with every cell no valid segment can see set to `value`."""
    k = call.k_store.clone()
    v = call.v_store.clone()
    needed = np.zeros((call.rows, call.cols), dtype=bool)
    for seg in np.asarray(call.seq_info, dtype=np.int64):
        if O.segment_status(seg, call.T, call.rows, call.cols, call.window):
            continue
        _, q_len, col, kv_end = (int(x) for x in seg)
        span = O.needed_span(q_len, kv_end, call.window)
        for j in range(kv_end - span, kv_end):
            needed[j % call.rows, col] = True
    mask = torch.from_numpy(~needed)
    k[mask] = value
    v[mask] = value
    return k, v


def digits16(j, n=5):
    return [(j >> (4 * d)) & 15 for d in range(n)]


def probe_call(call, sign):
    """Index-set probe inputs: K = V of position j spell j in base 16 over dims 0..4,
    q = +-16^d there, scale 64, so each row's output spells its last (sign +1) or first
    (sign -1) visible position exactly."""
    q = torch.zeros_like(call.q)
    for d in range(5):
        q[:, :, d] = sign * float(16 ** d)
    k = torch.zeros_like(call.k_store)
    for seg in np.asarray(call.seq_info, dtype=np.int64):
        if O.segment_status(seg, call.T, call.rows, call.cols, call.window):
            continue
        _, q_len, col, kv_end = (int(x) for x in seg)
        if q_len <= 0:
            continue
        span = O.needed_span(q_len, kv_end, call.window)
        js = np.arange(kv_end - span, kv_end)
        dig = torch.tensor([digits16(int(j)) for j in js], dtype=torch.bfloat16)
        k[torch.from_numpy(js % call.rows), col, :, :5] = dig[:, None, :]
    return q, k


def decode_probe(out: torch.Tensor):
    d = out[:, :, :5].double().cpu().numpy()
    return np.rint(d).astype(np.int64) @ (16 ** np.arange(5))
