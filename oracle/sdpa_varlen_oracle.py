"""Plain fp64 CPU oracle for length-aware GQA attention over a per-sequence KV column store.

TEST INFRASTRUCTURE. Only the tests, the smoke check of the package entry file and the
CPU-baseline leg of the bench may import or call this module.  The product path (the
CUDA library and its Python binding) never imports it and shares no code with it.

What is computed, and where the pages say so
--------------------------------------------
Sources are the pages' own titles:

* [A] "[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns"
  (#24072), PR description: each resident sequence owns one column of a
  [rows, cols, H, D] store; a device segment table seq_info Int32[S, 4] =
  (q_start, q_len, col, kv_end) says which packed query rows belong to which column and
  how long that sequence is; causal, non-causal, sliding window and ring storage, GQA;
  rows no segment covers are zeroed.
* [B] the #24074 commit message in that stack (LowerOffGraphKVPass batched-sequence
  manifest): the step's keys are written to slot (position % rows) * columns + col
  *before* the attention reads the store ("write then attend").
* [C] the #24073 commit message in that stack (CudaBatchedSequenceCache): the last
  column of [rows, max_seqs + 1, H, D] is scratch; ring layers hold
  min(capacity, window + max_write - 1) rows.
* [D] "[CUDA] Use Triton TMA for long-context causal prefill" (#22193), Summary:
  fully masked rows keep finite outputs.

Readings taken where the pages are silent (each is listed in the design notes):

1. Query row i of segment (q_start, q_len, col, kv_end) is packed row q_start + i and
   sits at position p = kv_end - q_len + i: the step's queries are the last q_len
   positions, already written into the store [B].
2. Visible keys: j < kv_end; causal adds j <= p; a window W > 0 adds j > p - W, i.e.
   W keys counting the query's own.  This is the only reading under which the ring
   size window + max_write - 1 of [C] holds exactly the keys one step can see.
   The window bound applies to non-causal calls too.
3. Position j of column col is read from store row j % rows (ring storage, [B]).
4. GQA: query head h reads KV head h // (Hq / Hkv).
5. scores = scale * q . k; softmax with base e; output = sum_j softmax_j * v_j.
6. An empty visible set gives 0 (a finite output [D]); a row no valid segment covers
   gives 0 [A].
7. A segment is invalid (skipped; its rows count as uncovered; a status bit is set) when
   q_len < 0, q_start < 0, q_start + q_len > T, col outside [0, cols), kv_end < 0, or
   when the keys its rows see span more than `rows` store rows (a ring would already
   have overwritten one of them).  When two valid segments cover a common row, both
   are overlapping: the overlap bit is set and every row of either segment has an
   unspecified output.

The arithmetic is fp64 from the exact upcast of the bf16 inputs.
"""

from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np

# Status bits (same values as the C interface's, written out independently here).
SEG_BAD_QRANGE = 1   # q_len < 0, q_start < 0 or q_start + q_len > T
SEG_BAD_COL = 2      # col outside [0, cols)
SEG_BAD_KV = 4       # kv_end < 0
SEG_SPAN = 8         # visible keys span more than `rows` store rows
SEG_OVERLAP = 16     # two valid segments cover the same packed row

UNCOVERED = -1
OVERLAPPED = -2


def _as_f64(x) -> np.ndarray:
    """Exact upcast of a bf16 (or any float) tensor/array to a float64 ndarray."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def row_interval(i: int, q_len: int, kv_end: int, causal: bool, window: int) -> Tuple[int, int]:
    """Visible key positions [lo, hi) of query row i of a segment (readings 1 and 2).

    Returns an interval with hi <= lo when the row sees nothing.
    """
    p = kv_end - q_len + i
    hi = min(p + 1, kv_end) if causal else kv_end
    lo = max(0, p - window + 1) if window > 0 else 0
    return lo, hi


def kv_head(h: int, group: int) -> int:
    """KV head read by query head h (reading 4)."""
    return h // group


def store_row(j, rows: int):
    """Store row holding logical position j of a column (reading 3)."""
    return j % rows


def needed_span(q_len: int, kv_end: int, window: int) -> int:
    """Number of consecutive positions the rows of one segment see together.

    The union of the rows' intervals is [lo of row 0, kv_end) whether or not the call
    is causal (row 0 has the smallest lower bound and some row reaches kv_end).
    """
    if q_len <= 0 or kv_end <= 0:
        return 0
    lo0, _ = row_interval(0, q_len, kv_end, False, window)
    return kv_end - lo0


def segment_status(seg, T: int, rows: int, cols: int, window: int) -> int:
    """Status bits of one segment (reading 7); 0 means valid."""
    q_start, q_len, col, kv_end = (int(x) for x in seg)
    bits = 0
    if q_len < 0 or q_start < 0 or q_start + q_len > T:
        bits |= SEG_BAD_QRANGE
    if col < 0 or col >= cols:
        bits |= SEG_BAD_COL
    if kv_end < 0:
        bits |= SEG_BAD_KV
    if bits == 0 and needed_span(q_len, kv_end, window) > rows:
        bits |= SEG_SPAN
    return bits


def segment_modes(seq_info, causal: bool, window: int, seg_mode=None):
    """Per segment (causal, window): the call's pair for every segment, or the rows of
    ``seg_mode`` [S, 2] when given (a per-segment mask mode, so that causal target segments
    and non-causal draft blocks can share one call)."""
    n = len(np.asarray(seq_info, dtype=np.int64).reshape(-1, 4))
    if seg_mode is None:
        return [(bool(causal), int(window))] * n
    m = np.asarray(seg_mode, dtype=np.int64).reshape(-1, 2)
    assert len(m) == n
    return [(bool(c), int(w)) for c, w in m]


def visible_interval(seq_info, T: int, causal: bool, window: int, rows: int, cols: int, seg_mode=None):
    """Per packed row: (segment id, lo, hi, status).

    seg_id[t] is the index of the valid segment covering row t, UNCOVERED when none
    does and OVERLAPPED when t belongs to a segment that shares a row with another
    valid segment (reading 7).  lo/hi are the row's visible positions (hi <= lo:
    empty); both are 0 for uncovered and overlapped rows.  status is the OR of every
    segment's bits plus SEG_OVERLAP.
    """
    modes = segment_modes(seq_info, causal, window, seg_mode)
    seq_info = np.asarray(seq_info, dtype=np.int64).reshape(-1, 4)
    seg_id = np.full(T, UNCOVERED, dtype=np.int64)
    lo = np.zeros(T, dtype=np.int64)
    hi = np.zeros(T, dtype=np.int64)
    status = 0
    owners = [[] for _ in range(T)]
    valid = []
    for s, seg in enumerate(seq_info):
        bits = segment_status(seg, T, rows, cols, modes[s][1])
        status |= bits
        if bits:
            continue
        valid.append(s)
        q_start, q_len = int(seg[0]), int(seg[1])
        for t in range(q_start, q_start + q_len):
            owners[t].append(s)
    overlapping = set()
    for t in range(T):
        if len(owners[t]) > 1:
            overlapping.update(owners[t])
    if overlapping:
        status |= SEG_OVERLAP
    for s in valid:
        q_start, q_len, _, kv_end = (int(x) for x in seq_info[s])
        for i in range(q_len):
            t = q_start + i
            if s in overlapping:
                seg_id[t] = OVERLAPPED
                lo[t] = hi[t] = 0
                continue
            seg_id[t] = s
            lo[t], hi[t] = row_interval(i, q_len, kv_end, modes[s][0], modes[s][1])
    return seg_id, lo, hi, status


def sdpa_varlen(q, k_store, v_store, seq_info, causal: bool, window: int, scale: float,
                rows_subset: Optional[Iterable[int]] = None, seg_mode=None):
    """Length-aware GQA attention over a column store, in fp64.

    q: [T, Hq, D]; k_store, v_store: [rows, cols, Hkv, D]; seq_info: [S, 4].
    Returns (out [T, Hq, D] float64, seg_id [T], status).  Rows outside
    ``rows_subset`` (when given) are left at 0 and not computed.  ``seg_mode`` [S, 2]
    (optional) gives each segment its own (causal, window) in place of the call's.
    """
    qf = _as_f64(q)
    T, Hq, D = qf.shape
    rows, cols, Hkv, Dk = k_store.shape
    assert Dk == D and tuple(v_store.shape) == tuple(k_store.shape)
    assert Hq % Hkv == 0
    group = Hq // Hkv
    seq_info = np.asarray(seq_info, dtype=np.int64).reshape(-1, 4)
    modes = segment_modes(seq_info, causal, window, seg_mode)
    seg_id, lo, hi, status = visible_interval(seq_info, T, causal, window, rows, cols, seg_mode)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    wanted = None if rows_subset is None else set(int(t) for t in rows_subset)

    for s, (q_start, q_len, col, kv_end) in enumerate(seq_info):
        rows_of_s = [t for t in range(q_start, q_start + max(q_len, 0))
                     if 0 <= t < T and seg_id[t] == s and (wanted is None or t in wanted)]
        if not rows_of_s:
            continue
        # Upcast the keys/values this segment can see once: positions [u_lo, kv_end).
        u_lo = kv_end - needed_span(q_len, kv_end, modes[s][1])
        pos = np.arange(u_lo, kv_end)
        phys = store_row(pos, rows)
        Kc = _as_f64(k_store[phys, col])                     # [n, Hkv, D]
        Vc = _as_f64(v_store[phys, col])
        for t in rows_of_s:
            a, b = int(lo[t]), int(hi[t])
            if b <= a:
                continue                                     # empty set: 0 (reading 6)
            for hk in range(Hkv):
                heads = [h for h in range(Hq) if kv_head(h, group) == hk]
                K = Kc[a - u_lo:b - u_lo, hk, :]             # [n, D]
                V = Vc[a - u_lo:b - u_lo, hk, :]
                sc = scale * (qf[t, heads, :] @ K.T)         # [group, n]   (reading 5)
                sc = sc - sc.max(axis=1, keepdims=True)
                e = np.exp(sc)
                w = e / e.sum(axis=1, keepdims=True)
                out[t, heads, :] = w @ V
    return out, seg_id, status


def sdpa_causal_prefill(q, k, v, scale: float, rows_subset: Optional[Iterable[int]] = None):
    """Dense causal GQA attention, queries being the last Lq of Lkv positions.

    q: [Lq, Hq, D]; k, v: [Lkv, Hkv, D].  A [Lkv, Hkv, D] tensor is a flat store with
    one column, so this is the one-segment case (0, Lq, 0, Lkv) of ``sdpa_varlen``.
    """
    Lq = q.shape[0]
    Lkv = k.shape[0]
    seq_info = np.array([[0, Lq, 0, Lkv]], dtype=np.int64)
    out, _, _ = sdpa_varlen(q, k[:, None], v[:, None], seq_info, True, 0, scale, rows_subset)
    return out


def kv_append(k_store, v_store, k_new, v_new, seq_info, window: int):
    """The step's keys and values written into the column store before attention [B].

    k_store, v_store: [rows, cols, Hkv, D]; k_new, v_new: [T, Hkv, D] (packed rows).
    Row q_start + i of a live segment (valid and not overlapping, reading 7) holds
    position p = kv_end - q_len + i (reading 1) and is written to store row p % rows
    (reading 3) of the segment's column, every KV head.  Rows with p < 0, rows of
    invalid or overlapping segments and rows no segment covers write nothing.  Returns
    new copies of the stores (same dtype); the inputs are not modified.
    """
    import torch

    T = k_new.shape[0]
    rows, cols = k_store.shape[0], k_store.shape[1]
    seg_id, _, _, _ = visible_interval(seq_info, T, True, window, rows, cols)
    k_out = k_store.clone()
    v_out = v_store.clone()
    seq_info = np.asarray(seq_info, dtype=np.int64).reshape(-1, 4)
    for s, (q_start, q_len, col, kv_end) in enumerate(seq_info):
        for i in range(max(int(q_len), 0)):
            t = int(q_start) + i
            if not (0 <= t < T) or seg_id[t] != s:
                continue
            p = int(kv_end) - int(q_len) + i
            if p < 0:
                continue
            k_out[store_row(p, rows), int(col)] = k_new[t]
            v_out[store_row(p, rows), int(col)] = v_new[t]
    assert isinstance(k_out, torch.Tensor)
    return k_out, v_out


def seq_clone(k_store, v_store, src_col: int, dst_col: int, n: int):
    """Column dst_col takes over the first n positions of column src_col (the #24073 commit
    message in the stack of [A]: seq_clone, a device copy of the source prefix).

    Position j lives in store row j % rows (reading 3), so a ring only holds the last
    `rows` of them: positions [max(0, n - rows), n) are copied, each from its row of the
    source column to the same row of the destination, every KV head, K and V.  Rows the
    prefix does not reach keep their contents.  Returns new copies of the stores.
    """
    rows = k_store.shape[0]
    k_out = k_store.clone()
    v_out = v_store.clone()
    for j in range(max(0, n - rows), n):
        r = store_row(j, rows)
        k_out[r, dst_col] = k_store[r, src_col]
        v_out[r, dst_col] = v_store[r, src_col]
    return k_out, v_out


def useful_flops(seq_info, T: int, Hq: int, D: int, causal: bool, window: int, rows: int, cols: int) -> int:
    """4 * D * Hq * sum over covered rows of |visible set| (QK^T and PV multiply-adds)."""
    _, lo, hi, _ = visible_interval(seq_info, T, causal, window, rows, cols)
    n = int(np.maximum(hi - lo, 0).sum())
    return 4 * D * Hq * n


def useful_kv_bytes(seq_info, T: int, Hkv: int, D: int, window: int, rows: int, cols: int,
                    elem_bytes: int = 2) -> int:
    """Bytes of K and V that the valid segments must read once: the union of their rows'
    visible sets, per KV head, for K and for V."""
    seq_info = np.asarray(seq_info, dtype=np.int64).reshape(-1, 4)
    total = 0
    for seg in seq_info:
        if segment_status(seg, T, rows, cols, window):
            continue
        _, q_len, _, kv_end = (int(x) for x in seg)
        total += needed_span(q_len, kv_end, window) * Hkv * D * elem_bytes * 2
    return total
