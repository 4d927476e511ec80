"""Pins of the oracle's KV append (the step's keys and values written into the column store
before the attention reads it: "[executorch][cuda] Add a length-aware Triton SDPA over
per-sequence KV columns", #24074 commit message, slot (position % rows) * columns + col).

Each check rests on something other than the oracle's own formula: a slice assignment, the
flat/ring folding of positions, torch's dense attention, and invariants."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import sdpa_varlen_oracle as O  # noqa: E402

pytestmark = pytest.mark.filterwarnings("ignore")


def _store(rows, cols, Hkv, D, fill=float("nan")):
    return torch.full((rows, cols, Hkv, D), fill, dtype=torch.bfloat16)


def _new(T, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16),
            torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16))


def test_one_segment_fills_its_column_prefix():
    k0, v0 = _store(40, 3, 2, 8), _store(40, 3, 2, 8)
    kn, vn = _new(12, 2, 8, 1)
    k, v = O.kv_append(k0, v0, kn, vn, [[0, 12, 1, 12]], 0)
    assert torch.equal(k[:12, 1], kn) and torch.equal(v[:12, 1], vn)
    assert torch.isnan(k[12:, 1].float()).all() and torch.isnan(k[:, 0].float()).all()
    assert torch.isnan(k[:, 2].float()).all() and torch.isnan(v[12:, 1].float()).all()


def test_decode_rows_land_at_their_positions():
    # S sequences, one query each: row i goes to position kv_end_i - 1 of column i
    rng = np.random.default_rng(3)
    S, rows = 6, 50
    kv = rng.integers(1, rows + 1, size=S)
    seq = np.array([[i, 1, i, int(kv[i])] for i in range(S)])
    kn, vn = _new(S, 2, 8, 2)
    k, v = O.kv_append(_store(rows, S, 2, 8), _store(rows, S, 2, 8), kn, vn, seq, 0)
    for i in range(S):
        assert torch.equal(k[int(kv[i]) - 1, i], kn[i]) and torch.equal(v[int(kv[i]) - 1, i], vn[i])
    assert int((~torch.isnan(k.float())).sum()) == S * 2 * 8


def test_ring_store_is_the_flat_store_folded():
    # the same table appended to a flat store and to a ring of R rows: every written
    # position p of the flat store reappears at ring row p % R
    R, window = 9, 6
    seq = np.array([[0, 4, 0, 23], [4, 3, 1, 5], [7, 4, 2, 40]])  # spans 9, 8, 9 <= R
    kn, vn = _new(12, 1, 4, 5)  # row 11 uncovered
    kf, _ = O.kv_append(_store(64, 3, 1, 4), _store(64, 3, 1, 4), kn, vn, seq, window)
    kr, _ = O.kv_append(_store(R, 3, 1, 4), _store(R, 3, 1, 4), kn, vn, seq, window)
    written = ~torch.isnan(kf.float()).all(dim=(2, 3))
    for p, c in zip(*torch.nonzero(written, as_tuple=True)):
        assert torch.equal(kr[int(p) % R, int(c)], kf[int(p), int(c)])
    assert int(written.sum()) == int((~torch.isnan(kr.float()).all(dim=(2, 3))).sum()) == 11


def test_invalid_overlapping_uncovered_and_negative_positions_write_nothing():
    seq = np.array([
        [0, 3, 0, 10],   # valid
        [3, 2, 5, 10],   # column out of range
        [5, 2, 1, 10],   # overlaps the next one: both dropped
        [6, 2, 2, 10],
        [9, 4, 3, 2],    # kv_end < q_len: positions -2, -1, 0, 1 -> only 0 and 1 written
    ])
    kn, vn = _new(16, 1, 4, 7)   # rows 8 and 13..15 are uncovered
    k, _ = O.kv_append(_store(12, 4, 1, 4), _store(12, 4, 1, 4), kn, vn, seq, 0)
    filled = ~torch.isnan(k.float()).all(dim=(2, 3))
    expect = torch.zeros(12, 4, dtype=torch.bool)
    expect[7:10, 0] = True
    expect[0:2, 3] = True
    assert torch.equal(filled, expect)
    assert torch.equal(k[0, 3], kn[11]) and torch.equal(k[1, 3], kn[12])


def test_append_then_attend_equals_dense_attention_over_the_new_rows():
    # non-causal, kv_end = q_len: after the append the segment sees exactly the new rows,
    # so the result is plain softmax attention over them (torch, fp64); the store starts
    # as NaN, so any cell the append missed would poison the output
    T, Hq, Hkv, D = 10, 4, 2, 16
    kn, vn = _new(T, Hkv, D, 11)
    q = torch.randn(T, Hq, D, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    seq = np.array([[0, T, 1, T]])
    k, v = O.kv_append(_store(32, 2, Hkv, D), _store(32, 2, Hkv, D), kn, vn, seq, 0)
    out, _, _ = O.sdpa_varlen(q, k, v, seq, False, 0, 0.25)
    qd = q.double().transpose(0, 1)
    kd = kn.double().repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
    vd = vn.double().repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=0.25).transpose(0, 1)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_append_is_idempotent_and_leaves_inputs_alone():
    seq = np.array([[0, 5, 0, 9], [5, 3, 1, 3]])
    kn, vn = _new(8, 2, 8, 13)
    k0, v0 = _store(16, 2, 2, 8, 0.5), _store(16, 2, 2, 8, -0.5)
    k1, v1 = O.kv_append(k0, v0, kn, vn, seq, 0)
    k2, v2 = O.kv_append(k1, v1, kn, vn, seq, 0)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(k0, torch.full_like(k0, 0.5)) and torch.equal(v0, torch.full_like(v0, -0.5))


# seq_clone: column dst takes over the first n positions of column src (#24073 commit message)

def test_clone_of_a_short_prefix_copies_that_many_rows():
    g = torch.Generator().manual_seed(21)
    k0 = torch.randn(16, 4, 2, 8, generator=g).to(torch.bfloat16)
    v0 = torch.randn(16, 4, 2, 8, generator=g).to(torch.bfloat16)
    k, v = O.seq_clone(k0, v0, 1, 3, 5)
    assert torch.equal(k[:5, 3], k0[:5, 1]) and torch.equal(v[:5, 3], v0[:5, 1])
    assert torch.equal(k[5:, 3], k0[5:, 3]) and torch.equal(k[:, :3], k0[:, :3])


def test_clone_of_a_wrapped_ring_copies_the_whole_column():
    # n > rows: every row holds a position of the prefix, so the whole column moves
    g = torch.Generator().manual_seed(22)
    k0 = torch.randn(7, 3, 1, 4, generator=g).to(torch.bfloat16)
    v0 = torch.randn(7, 3, 1, 4, generator=g).to(torch.bfloat16)
    k, v = O.seq_clone(k0, v0, 0, 2, 30)
    assert torch.equal(k[:, 2], k0[:, 0]) and torch.equal(v[:, 2], v0[:, 0])
    assert torch.equal(k[:, :2], k0[:, :2])


def test_clone_then_attend_matches_the_source_sequence():
    # a sequence cloned into a new column attends exactly like the original one
    g = torch.Generator().manual_seed(23)
    rows, Hkv, D = 20, 2, 8
    k0 = torch.randn(rows, 3, Hkv, D, generator=g).to(torch.bfloat16)
    v0 = torch.randn(rows, 3, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(3, 4, D, generator=g).to(torch.bfloat16)
    k, v = O.seq_clone(k0, v0, 0, 2, 26)
    a, _, _ = O.sdpa_varlen(q, k, v, [[0, 3, 0, 26]], True, 10, 0.3)
    b, _, _ = O.sdpa_varlen(q, k, v, [[0, 3, 2, 26]], True, 10, 0.3)
    np.testing.assert_array_equal(a, b)
