"""Pins of the oracle's per-segment mask mode (each segment its own (causal, window), so that
causal target segments and non-causal draft blocks share one call: a per-segment mode of the
"[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns" stack, whose
#24074 manifest carries `causal` per model and whose DFlash drafts are non-causal).

A table of uniform modes must reduce to the call-level oracle (pinned on its own in
test_oracle_pins.py); a mixed table must equal the call-level results of its two halves run
as separate calls; validity uses each segment's own window."""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import sdpa_varlen_oracle as O  # noqa: E402

pytestmark = pytest.mark.filterwarnings("ignore")


def _inputs(T, Hq, Hkv, D, rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(T, Hq, D, generator=g).to(torch.bfloat16),
            torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16),
            torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16))


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 3), (False, 5)])
def test_uniform_modes_reduce_to_the_call_level_mask(causal, window):
    q, k, v = _inputs(20, 4, 2, 8, 40, 3, 1)
    seq = np.array([[0, 5, 0, 17], [6, 3, 1, 3], [10, 7, 2, 30], [17, 2, 0, 1]])
    modes = np.array([[int(causal), window]] * len(seq))
    a, sa, ta = O.sdpa_varlen(q, k, v, seq, causal, window, 0.35)
    b, sb, tb = O.sdpa_varlen(q, k, v, seq, not causal, window + 2, 0.35, seg_mode=modes)
    np.testing.assert_array_equal(a, b)
    assert np.array_equal(sa, sb) and ta == tb


def test_a_mixed_table_equals_its_halves_run_as_separate_calls():
    q, k, v = _inputs(32, 4, 1, 8, 64, 4, 2)
    target = np.array([[0, 4, 0, 50], [4, 2, 1, 20]])      # causal, window 8
    draft = np.array([[16, 6, 2, 30], [24, 5, 3, 12]])     # non-causal, no window
    seq = np.concatenate([target, draft])
    modes = np.array([[1, 8], [1, 8], [0, 0], [0, 0]])
    mixed, seg_id, st = O.sdpa_varlen(q, k, v, seq, True, 0, 0.4, seg_mode=modes)
    a, _, _ = O.sdpa_varlen(q, k, v, target, True, 8, 0.4)
    b, _, _ = O.sdpa_varlen(q, k, v, draft, False, 0, 0.4)
    np.testing.assert_array_equal(mixed[:16], a[:16])
    np.testing.assert_array_equal(mixed[16:], b[16:])
    assert st == 0 and (seg_id[6:16] == O.UNCOVERED).all()


def test_validity_uses_each_segments_own_window():
    # on a 12-row ring, kv_end 40 is fine under a window of 6 (span 3 + 6 - 1 = 8) and
    # invalid without one (span 40)
    seq = np.array([[0, 3, 0, 40], [3, 3, 1, 40]])
    _, _, _, st_w = O.visible_interval(seq, 6, True, 0, 12, 2, seg_mode=[[1, 6], [1, 6]])
    _, _, _, st_mixed = O.visible_interval(seq, 6, True, 0, 12, 2, seg_mode=[[1, 6], [1, 0]])
    assert st_w == 0 and st_mixed == O.SEG_SPAN
