"""Seeded synthetic inputs for length-aware GQA attention over a KV column store.

This module only draws numbers: it holds none of the attention arithmetic, no mask
or interval logic and nothing shared with either the CUDA path or the CPU oracle.
Both sides (and the bench) build their inputs here, so that a parity test feeds the
same tensors to both.

Recipe (the same for every workload):
  * integer draws (segment lengths, KV ends) come first, from
    ``numpy.random.default_rng(seed)``, in the order the workload lists them;
  * then every bf16 tensor, in the order q, k_store, v_store (and, for the mixed
    step, the ring store pair before the flat store pair), from
    ``torch.randn(shape, generator=torch.Generator().manual_seed(seed))`` in fp32,
    rounded to bf16 (round-to-nearest-even by ``Tensor.to``);
  * the whole store is filled i.i.d., including the scratch column and cells no
    segment can see.

Shapes follow the workloads measured on the pages: "[CUDA] Use Triton TMA for
long-context causal prefill" (Operator-level performance table: B=1, Hq=16, Hkv=2,
D in {64, 128}, Lq/Lkv 512/16,384 and 4,096/131,072) and "[executorch][cuda] Add a
length-aware Triton SDPA over per-sequence KV columns" (column store
[rows, cols, H, D] with a trailing scratch column, ring rows
window + max_write - 1, segment table (q_start, q_len, col, kv_end)).
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass
class Call:
    """One attention call: packed queries against one column store."""

    T: int
    Hq: int
    Hkv: int
    D: int
    rows: int
    cols: int
    seq_info: np.ndarray  # int32 [S, 4] = (q_start, q_len, col, kv_end)
    causal: bool
    window: int
    scale: float
    q: torch.Tensor  # bf16 [T, Hq, D] (CPU)
    k_store: torch.Tensor  # bf16 [rows, cols, Hkv, D] (CPU)
    v_store: torch.Tensor  # bf16 [rows, cols, Hkv, D] (CPU)
    # Packed rows [row_begin, row_end) of the step this call owns (a mixed step runs one
    # call per store); q and seq_info are relative to row_begin.
    row_begin: int = 0
    row_end: Optional[int] = None
    # int32 [S, 2] = (causal, window) per segment, replacing causal / window when given
    seg_mode: Optional[np.ndarray] = None


@dataclasses.dataclass
class Workload:
    name: str
    calls: List[Call]
    description: str


def _randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _seq_info(rows_list) -> np.ndarray:
    a = np.asarray(rows_list, dtype=np.int64).reshape(-1, 4)
    return a.astype(np.int32)


def tiny_causal_prefill(seed: int = 0) -> Workload:
    """S=1, Hq=4, Hkv=1, D=64, q_len=kv_end=128, flat store [128, 1, 1, 64]."""
    T, Hq, Hkv, D, rows, cols = 128, 4, 1, 64, 128, 1
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    c = Call(T, Hq, Hkv, D, rows, cols, _seq_info([(0, 128, 0, 128)]), True, 0,
             1.0 / math.sqrt(D), q, k, v)
    return Workload("tiny_causal_prefill_d64", [c], "S=1 Hq=4 Hkv=1 D=64 q_len=kv_end=128 causal")


def long_causal_prefill(D: int, Lq: int, Lkv: int, seed: int = 0, Hq: int = 16, Hkv: int = 2) -> Workload:
    """Dense causal GQA prefill as one segment: queries are the last Lq of Lkv positions."""
    T, rows, cols = Lq, Lkv, 1
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    c = Call(T, Hq, Hkv, D, rows, cols, _seq_info([(0, Lq, 0, Lkv)]), True, 0,
             1.0 / math.sqrt(D), q, k, v)
    return Workload(f"causal_gqa_prefill_d{D}_q{Lq}_kv{Lkv}", [c],
                    f"S=1 Hq={Hq} Hkv={Hkv} D={D} Lq={Lq} Lkv={Lkv} causal")


def batched_decode(seed: int = 0, S: int = 32, Hq: int = 16, Hkv: int = 2, D: int = 128,
                   rows: int = 8192) -> Workload:
    """S sequences, one query each; column S of the store is scratch."""
    rng = np.random.default_rng(seed)
    kv_end = rng.integers(1, rows + 1, size=S)
    T, cols = S, S + 1
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    si = _seq_info([(i, 1, i, int(kv_end[i])) for i in range(S)])
    c = Call(T, Hq, Hkv, D, rows, cols, si, True, 0, 1.0 / math.sqrt(D), q, k, v)
    return Workload(f"splitk_decode_s{S}_d{D}", [c],
                    f"S={S} q_len=1 Hq={Hq} Hkv={Hkv} D={D} store [{rows},{cols},{Hkv},{D}] causal")


def mixed_step(seed: int = 0, n_target: int = 8, n_draft: int = 8, Hq: int = 32, Hkv: int = 8,
               D: int = 128, window: int = 4096, max_write: int = 16, flat_rows: int = 8192,
               kv_lo: int = 2000, kv_hi: int = 60000, T: int = 256) -> Workload:
    """Sliding-window targets on a ring store plus non-causal draft blocks on a flat store.

    Rows [0, T/2) hold the targets, packed from row 0 (the rows after the last
    target stay uncovered); rows [T/2, T) hold the draft blocks of max_write rows.  The
    step is two calls, one per store, each owning its half of the packed rows: its q is
    a view of those rows and its q_start values count from the half's first row.
    """
    rng = np.random.default_rng(seed)
    q_len_t = rng.integers(1, max_write + 1, size=n_target)
    kv_end_t = rng.integers(kv_lo, kv_hi + 1, size=n_target)
    kv_end_d = rng.integers(max_write, flat_rows + 1, size=n_draft)
    ring_rows = window + max_write - 1
    cols = max(n_target, n_draft) + 1
    half = T // 2
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, Hq, D))
    rk = _randn_bf16(gen, (ring_rows, cols, Hkv, D))
    rv = _randn_bf16(gen, (ring_rows, cols, Hkv, D))
    fk = _randn_bf16(gen, (flat_rows, cols, Hkv, D))
    fv = _randn_bf16(gen, (flat_rows, cols, Hkv, D))
    segs_a, start = [], 0
    for k in range(n_target):
        segs_a.append((start, int(q_len_t[k]), k, int(kv_end_t[k])))
        start += int(q_len_t[k])
    # q_start of each call is relative to the first packed row the call owns
    segs_b = [(max_write * k, max_write, k, int(kv_end_d[k])) for k in range(n_draft)]
    scale = 1.0 / math.sqrt(D)
    a = Call(half, Hq, Hkv, D, ring_rows, cols, _seq_info(segs_a), True, window, scale, q[:half],
             rk, rv, row_begin=0, row_end=half)
    b = Call(T - half, Hq, Hkv, D, flat_rows, cols, _seq_info(segs_b), False, 0, scale, q[half:],
             fk, fv, row_begin=half, row_end=T)
    return Workload("mixed_swa_ring_draft_step", [a, b],
                    f"T={T} Hq={Hq} Hkv={Hkv} D={D}: {n_target} causal W={window} ring segments "
                    f"(rows {ring_rows}) + {n_draft} non-causal {max_write}-row draft blocks")


def mixed_step_one_store(seed: int = 0, n_target: int = 8, n_draft: int = 8, Hq: int = 32, Hkv: int = 8,
                         D: int = 128, window: int = 4096, max_write: int = 16, kv_lo: int = 2000,
                         kv_hi: int = 60000, T: int = 256) -> Workload:
    """The mixed step of ``mixed_step`` as one call over one ring store: the targets (causal,
    window W, kv_end far past the ring) and the draft blocks (non-causal, no window, kv_end
    within the ring) each carry their own mode in ``seg_mode``.

    Rows [0, T/2) hold the targets, packed from row 0; draft block k holds rows
    T/2 + max_write * k onwards.  Column k holds target k, column n_target + k draft k.
    """
    rng = np.random.default_rng(seed)
    q_len_t = rng.integers(1, max_write + 1, size=n_target)
    kv_end_t = rng.integers(kv_lo, kv_hi + 1, size=n_target)
    rows = window + max_write - 1
    kv_end_d = rng.integers(max_write, rows + 1, size=n_draft)
    cols = n_target + n_draft + 1
    half = T // 2
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (T, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    segs, modes, start = [], [], 0
    for i in range(n_target):
        segs.append((start, int(q_len_t[i]), i, int(kv_end_t[i])))
        modes.append((1, window))
        start += int(q_len_t[i])
    for i in range(n_draft):
        segs.append((half + max_write * i, max_write, n_target + i, int(kv_end_d[i])))
        modes.append((0, 0))
    c = Call(T, Hq, Hkv, D, rows, cols, _seq_info(segs), True, 0, 1.0 / math.sqrt(D), q, k, v,
             seg_mode=np.array(modes, dtype=np.int32))
    return Workload("mixed_swa_ring_draft_step_one_store", [c],
                    f"T={T} Hq={Hq} Hkv={Hkv} D={D}: {n_target} causal W={window} segments + {n_draft} "
                    f"non-causal {max_write}-row draft blocks on one {rows}-row ring store, one launch "
                    f"(per-segment modes)")


def ring_window_prefill(seed: int = 0, Hq: int = 16, Hkv: int = 2, D: int = 128, window: int = 4096,
                        q_len: int = 2048, kv_end: int = 60000) -> Workload:
    """A long sliding-window prefill chunk on a ring store: one segment of q_len queries whose
    keys [kv_end - q_len - window + 1, kv_end) wrap around a ring of window + q_len - 1 rows
    (the ring size of "[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV
    columns", #24073 commit: window + max_write - 1, with max_write = q_len).  Column 1 is the
    scratch column."""
    rows, cols = window + q_len - 1, 2
    gen = torch.Generator().manual_seed(seed)
    q = _randn_bf16(gen, (q_len, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    c = Call(q_len, Hq, Hkv, D, rows, cols, _seq_info([(0, q_len, 0, kv_end)]), True, window,
             1.0 / math.sqrt(D), q, k, v)
    return Workload(f"ring_window_prefill_w{window}_q{q_len}_kv{kv_end}_d{D}", [c],
                    f"S=1 Hq={Hq} Hkv={Hkv} D={D} causal W={window} q_len={q_len} kv_end={kv_end} "
                    f"on a ring of {rows} rows (keys wrap)")


def workload(index: int, seed: int = 0) -> Workload:
    """The measured shapes, in order: tiny, D=64 prefill, D=128 prefill, decode, mixed, the
    mixed step as one call with per-segment modes, a D=256 prefill, and a windowed prefill
    chunk on a ring store."""
    if index == 0:
        return tiny_causal_prefill(seed)
    if index == 1:
        return long_causal_prefill(64, 512, 16384, seed)
    if index == 2:
        return long_causal_prefill(128, 4096, 131072, seed)
    if index == 3:
        return batched_decode(seed)
    if index == 4:
        return mixed_step(seed)
    if index == 5:
        return mixed_step_one_store(seed)
    if index == 6:
        return long_causal_prefill(256, 4096, 32768, seed)
    if index == 7:
        return ring_window_prefill(seed)
    raise ValueError(f"no workload {index}")


def random_call(rng: np.random.Generator, *, D: int, Hq: int, Hkv: int, T: int, S: int,
                rows: int, cols: int, causal: bool, window: int, max_q: int, max_kv: int,
                gen_seed: int, allow_gaps: bool = True, distinct_cols: bool = False) -> Call:
    """A random segment table over packed rows (with uncovered gaps), for parity sweeps.

    Only draws numbers: segments are laid end to end with random gaps and kv_end is
    drawn in [0, max_kv] (beyond ``rows`` on a ring store).  Whether a drawn segment is
    valid is left to the code under test.
    """
    segs = []
    t = 0
    for s in range(S):
        if allow_gaps:
            t += int(rng.integers(0, 3))
        ql = int(rng.integers(0, max_q + 1))
        if t + ql > T:
            ql = max(0, T - t)
        ke = int(rng.integers(0, max_kv + 1))
        col = int(rng.integers(0, cols))
        if distinct_cols:
            col = s % cols  # one sequence per column
        segs.append((t, ql, col, ke))
        t += ql
    gen = torch.Generator().manual_seed(gen_seed)
    q = _randn_bf16(gen, (T, Hq, D))
    k = _randn_bf16(gen, (rows, cols, Hkv, D))
    v = _randn_bf16(gen, (rows, cols, Hkv, D))
    return Call(T, Hq, Hkv, D, rows, cols, _seq_info(segs), causal, window, 1.0 / math.sqrt(D), q, k, v)
