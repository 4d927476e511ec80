"""Pins for the CPU oracle: checks against things other than the oracle itself.

* a brute-force scalar restatement (per-element visibility predicates, ``math.exp``
  loops, and an aliasing test for the ring instead of the span formula) on an
  exhaustive seeded grid of tiny segment tables;
* the invariants the method fixes: one visible key returns its V row, constant V
  returns the constant, K = 0 averages the visible V rows, empty and uncovered rows
  are 0, a ring store equals the unrolled flat store;
* library special cases: ``torch.nn.functional.scaled_dot_product_attention`` in fp64
  on the CPU with an explicit boolean mask built here from the predicates, and with
  ``is_causal`` for q_len = kv_end;
* hand-worked golden cases (tests/golden/hand_cases.json);
* the ring size printed on the pages (window + max_write - 1) fixes the window reading;
* an index-set probe whose output spells the last (or first) visible position;
* planted mistakes in the oracle are caught by these pins.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import sdpa_varlen_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


# ---------------------------------------------------------------------------------------
# brute force: a second, scalar formulation written from the predicates
# ---------------------------------------------------------------------------------------

def _visible(j, p, kv_end, causal, W):
    if j < 0 or j >= kv_end:
        return False
    if causal and j > p:
        return False
    if W > 0 and j <= p - W:
        return False
    return True


def brute_force(q, K, V, seq_info, causal, W, scale):
    """q: nested list [T][Hq][D]; K, V: nested [rows][cols][Hkv][D]."""
    T, Hq, D = len(q), len(q[0]), len(q[0][0])
    rows, cols, Hkv = len(K), len(K[0]), len(K[0][0])
    group = Hq // Hkv
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(T)]
    owners = [[] for _ in range(T)]
    status = 0
    for s, (qs, ql, col, ke) in enumerate(seq_info):
        bad = 0
        if ql < 0 or qs < 0 or qs + ql > T:
            bad |= 1
        if not (0 <= col < cols):
            bad |= 2
        if ke < 0:
            bad |= 4
        if bad == 0:
            # every position some row of the segment sees
            seen = set()
            for i in range(ql):
                p = ke - ql + i
                for j in range(0, max(ke, 0)):
                    if _visible(j, p, ke, causal, W):
                        seen.add(j)
            # two seen positions in one store row: the ring overwrote one of them
            if len({j % rows for j in seen}) < len(seen):
                bad |= 8
        status |= bad
        if bad:
            continue
        for i in range(ql):
            owners[qs + i].append(s)
    overlapping = set()
    for t in range(T):
        if len(owners[t]) > 1:
            status |= 16
            overlapping.update(owners[t])
    for t in range(T):
        if len(owners[t]) != 1 or owners[t][0] in overlapping:
            continue
        qs, ql, col, ke = seq_info[owners[t][0]]
        p = ke - ql + (t - qs)
        vis = [j for j in range(max(ke, 0)) if _visible(j, p, ke, causal, W)]
        if not vis:
            continue
        for h in range(Hq):
            hk = h // group
            sc = [scale * sum(q[t][h][d] * K[j % rows][col][hk][d] for d in range(D)) for j in vis]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            z = sum(e)
            for d in range(D):
                out[t][h][d] = sum(e[n] * V[vis[n] % rows][col][hk][d] for n in range(len(vis))) / z
    return out, owners, status


def _rand_case(rng, *, T, Hq, Hkv, D, rows, cols, S, max_q, max_kv, allow_bad):
    segs = []
    t = 0
    for _ in range(S):
        t += int(rng.integers(0, 2))
        ql = int(rng.integers(0, max_q + 1))
        ke = int(rng.integers(0, max_kv + 1))
        col = int(rng.integers(0, cols))
        qs = t
        if allow_bad and rng.random() < 0.15:
            which = int(rng.integers(0, 5))
            if which == 0:
                ql = -1
            elif which == 1:
                qs = T - 1 if ql > 1 else T + 1
            elif which == 2:
                col = cols
            elif which == 3:
                ke = -2
            else:
                qs = max(0, t - 1)  # overlaps the previous segment
        segs.append((qs, ql, col, ke))
        t = max(t, qs + max(ql, 0))
    q = (rng.standard_normal((T, Hq, D))).round(3)
    K = (rng.standard_normal((rows, cols, Hkv, D))).round(3)
    V = (rng.standard_normal((rows, cols, Hkv, D))).round(3)
    return segs, q, K, V


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("W", [0, 1, 2, 3, 5])
def test_oracle_matches_brute_force_on_tiny_grid(causal, W):
    rng = np.random.default_rng(1000 + 10 * W + int(causal))
    for trial in range(40):
        rows = int(rng.choice([3, 5, 8, 12]))
        Hq, Hkv = [(1, 1), (2, 1), (4, 2), (3, 3)][trial % 4]
        T, D, cols = 10, 3, 3
        S = int(rng.integers(1, 4))
        segs, q, K, V = _rand_case(rng, T=T, Hq=Hq, Hkv=Hkv, D=D, rows=rows, cols=cols, S=S,
                                   max_q=4, max_kv=9, allow_bad=True)
        out, seg_id, status = O.sdpa_varlen(q, K, V, np.array(segs), causal, W, 0.7)
        ref, owners, ref_status = brute_force(q.tolist(), K.tolist(), V.tolist(), segs, causal, W, 0.7)
        assert status == ref_status, (segs, rows, W)
        overlapping = {s for t in range(T) if len(owners[t]) > 1 for s in owners[t]}
        for t in range(T):
            if any(s in overlapping for s in owners[t]):
                assert seg_id[t] == O.OVERLAPPED
                continue  # unspecified output
            np.testing.assert_allclose(out[t], np.array(ref[t]), rtol=1e-12, atol=1e-12,
                                       err_msg=f"segs={segs} rows={rows} W={W} causal={causal} t={t}")


# ---------------------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------------------

def _bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def test_single_visible_key_returns_its_v_row():
    # W=1 under causal masking leaves each row its own position only.
    rng = np.random.default_rng(0)
    rows, cols, Hkv, Hq, D = 7, 2, 2, 4, 8
    q, k, v = _bf16(rng, (5, Hq, D)), _bf16(rng, (rows, cols, Hkv, D)), _bf16(rng, (rows, cols, Hkv, D))
    seq = np.array([[0, 5, 1, 11]])  # positions 6..10 -> rows 6,0,1,2,3
    out, _, st = O.sdpa_varlen(q, k, v, seq, True, 1, 0.3)
    assert st == 0
    vf = v.double().numpy()
    for i in range(5):
        p = 11 - 5 + i
        for h in range(Hq):
            assert np.array_equal(out[i, h], vf[p % rows, 1, h // 2])


def test_constant_v_returns_the_constant():
    rng = np.random.default_rng(1)
    rows, cols, Hkv, Hq, D = 64, 1, 2, 8, 16
    q, k = _bf16(rng, (20, Hq, D)), _bf16(rng, (rows, cols, Hkv, D))
    v = torch.full((rows, cols, Hkv, D), 0.375, dtype=torch.bfloat16)
    for causal, W in [(True, 0), (False, 0), (True, 7), (False, 5)]:
        out, seg_id, _ = O.sdpa_varlen(q, k, v, np.array([[0, 20, 0, 50]]), causal, W, 0.25)
        np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-14)


def test_zero_keys_average_the_visible_values():
    rng = np.random.default_rng(2)
    rows, Hkv, Hq, D = 10, 1, 2, 4
    q = _bf16(rng, (3, Hq, D))
    k = torch.zeros((rows, 1, Hkv, D), dtype=torch.bfloat16)
    v = _bf16(rng, (rows, 1, Hkv, D))
    out, _, _ = O.sdpa_varlen(q, k, v, np.array([[0, 3, 0, 12]]), True, 4, 1.0)
    vf = v.double().numpy()[:, 0, 0]
    for i in range(3):
        p = 12 - 3 + i
        vis = [j % rows for j in range(p - 3, p + 1)]
        np.testing.assert_allclose(out[i, 0], vf[vis].mean(axis=0), rtol=1e-14, atol=1e-15)


def test_empty_and_uncovered_rows_are_exactly_zero():
    rng = np.random.default_rng(3)
    q, k, v = _bf16(rng, (8, 2, 4)), _bf16(rng, (6, 1, 1, 4)), _bf16(rng, (6, 1, 1, 4))
    # rows 0,1 uncovered; segment (2,4,0,2): positions -2,-1,0,1; rows 6,7 uncovered
    out, seg_id, _ = O.sdpa_varlen(q, k, v, np.array([[2, 4, 0, 2]]), True, 0, 1.0)
    for t in (0, 1, 2, 3, 6, 7):
        assert np.all(out[t] == 0.0)
    assert np.all(out[4] != 0.0) and np.all(out[5] != 0.0)
    assert list(seg_id) == [-1, -1, 0, 0, 0, 0, -1, -1]


def test_ring_store_equals_unrolled_flat_store():
    rng = np.random.default_rng(4)
    Hq, Hkv, D, W, q_len, kv_end = 4, 2, 8, 6, 3, 40
    rows = W + q_len - 1  # ring sized window + max_write - 1
    R_k, R_v = _bf16(rng, (rows, 1, Hkv, D)), _bf16(rng, (rows, 1, Hkv, D))
    q = _bf16(rng, (q_len, Hq, D))
    F_k = torch.full((kv_end, 1, Hkv, D), float("nan"), dtype=torch.bfloat16)
    F_v = F_k.clone()
    for j in range(kv_end - q_len - W + 1, kv_end):  # the positions the step can see
        F_k[j], F_v[j] = R_k[j % rows], R_v[j % rows]
    seq = np.array([[0, q_len, 0, kv_end]])
    for causal in (True, False):
        ring, _, st1 = O.sdpa_varlen(q, R_k, R_v, seq, causal, W, 0.5)
        flat, _, st2 = O.sdpa_varlen(q, F_k, F_v, seq, causal, W, 0.5)
        assert st1 == 0 and st2 == 0
        assert np.array_equal(ring, flat)


# ---------------------------------------------------------------------------------------
# library special cases
# ---------------------------------------------------------------------------------------

def _torch_ref(qf, kf, vf, mask, scale):
    """qf [T,Hq,D], kf/vf [n,Hkv,D] fp64; mask [T, n] bool (True = visible)."""
    Hq, Hkv = qf.shape[1], kf.shape[1]
    kk = kf.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    vv = vf.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    qq = qf.permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask[None], scale=scale)
    return o.permute(1, 0, 2)


def test_noncausal_full_equals_dense_softmax_attention():
    rng = np.random.default_rng(5)
    for Hq, Hkv, L in [(4, 1, 9), (8, 2, 33), (6, 3, 17)]:
        q, k, v = _bf16(rng, (L, Hq, 16)), _bf16(rng, (L, 1, Hkv, 16)), _bf16(rng, (L, 1, Hkv, 16))
        out, _, _ = O.sdpa_varlen(q, k, v, np.array([[0, L, 0, L]]), False, 0, 0.2)
        mask = torch.ones((L, L), dtype=torch.bool)
        ref = _torch_ref(q.double(), k[:, 0].double(), v[:, 0].double(), mask, 0.2)
        np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)
        # causal with q_len = kv_end is torch's top-left/bottom-right causal case alike
        outc, _, _ = O.sdpa_varlen(q, k, v, np.array([[0, L, 0, L]]), True, 0, 0.2)
        qq = q.double().permute(1, 0, 2)
        kk = k[:, 0].double().repeat_interleave(Hq // Hkv, 1).permute(1, 0, 2)
        vv = v[:, 0].double().repeat_interleave(Hq // Hkv, 1).permute(1, 0, 2)
        refc = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=0.2)
        np.testing.assert_allclose(outc, refc.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal,W", [(True, 0), (True, 5), (False, 0), (False, 4), (True, 1)])
def test_masked_library_attention_on_random_tables(causal, W):
    rng = np.random.default_rng(50 + W + 7 * causal)
    Hq, Hkv, D, rows, cols, T = 8, 2, 16, 24, 3, 40
    for trial in range(6):
        segs = []
        t = 0
        for _ in range(4):
            t += int(rng.integers(0, 3))
            ql = int(rng.integers(0, 8))
            ql = min(ql, T - t)
            ke = int(rng.integers(0, 40))
            segs.append((t, ql, int(rng.integers(0, cols)), ke))
            t += ql
        q, k, v = _bf16(rng, (T, Hq, D)), _bf16(rng, (rows, cols, Hkv, D)), _bf16(rng, (rows, cols, Hkv, D))
        out, seg_id, status = O.sdpa_varlen(q, k, v, np.array(segs), causal, W, 0.125)
        for s, (qs, ql, col, ke) in enumerate(segs):
            if ql == 0 or (seg_id[qs:qs + ql] != s).any():
                continue  # invalid segment: checked by the brute-force grid
            # the segment's visible positions, rebuilt from predicates over every position
            pos = np.arange(0, ke)
            p = ke - ql + np.arange(ql)
            vis = np.broadcast_to(pos[None, :] < ke, (ql, len(pos))).copy()
            if causal:
                vis &= pos[None, :] <= p[:, None]
            if W > 0:
                vis &= pos[None, :] > (p[:, None] - W)
            live = vis.any(axis=1)
            if not live.any():
                assert np.all(out[qs:qs + ql] == 0)
                continue
            kf = k[pos % rows, col].double()
            vf = v[pos % rows, col].double()
            ref = _torch_ref(q[qs:qs + ql].double()[live], kf, vf, torch.from_numpy(vis[live]), 0.125)
            np.testing.assert_allclose(out[qs:qs + ql][live], ref.numpy(), rtol=1e-11, atol=1e-12)
            assert np.all(out[qs:qs + ql][~live] == 0)


# ---------------------------------------------------------------------------------------
# hand-worked cases and the ring-size reading
# ---------------------------------------------------------------------------------------

def _case_tensors(c):
    T, Hq, Hkv, D, rows, cols = c["T"], c["Hq"], c["Hkv"], c["D"], c["rows"], c["cols"]
    q = np.zeros((T, Hq, D))
    k = np.zeros((rows, cols, Hkv, D))
    v = np.zeros((rows, cols, Hkv, D))
    for t, hs in c["q"].items():
        for h, vec in hs.items():
            q[int(t), int(h)] = vec
    for name, arr in (("k", k), ("v", v)):
        for r, cs in c[name].items():
            for col, hs in cs.items():
                for h, vec in hs.items():
                    arr[int(r), int(col), int(h)] = vec
    return q, k, v


def test_hand_worked_golden_cases():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 9
    for c in cases:
        q, k, v = _case_tensors(c)
        out, _, status = O.sdpa_varlen(q, k, v, np.array(c["seq_info"]), c["causal"], c["window"], c["scale"])
        assert status == c["status"], c["name"]
        for t, rowv in c["expected"].items():
            np.testing.assert_allclose(out[int(t)], np.array(rowv), rtol=1e-14, atol=1e-14, err_msg=c["name"])


def test_ring_size_on_the_pages_fits_one_step_exactly():
    # ring rows = window + max_write - 1 = 4096 + 16 - 1 (a ring layer of the batched
    # sequence cache); a 16-query step with W=4096 must fit in it, with no row to spare.
    W, max_write = 4096, 16
    rows = W + max_write - 1
    assert rows == 4111
    for kv_end in (4111, 4112, 60000):
        assert O.needed_span(max_write, kv_end, W) == rows
        assert O.segment_status((0, max_write, 0, kv_end), max_write, rows, 1, W) == 0
        assert O.segment_status((0, max_write, 0, kv_end), max_write, rows - 1, 1, W) == O.SEG_SPAN
    # under the other reading (j >= p - W, W + 1 keys) the same step would need 4112 rows
    p0, p_last = 60000 - 16, 60000 - 1
    assert (p_last + 1) - (p0 - W) == rows + 1


# ---------------------------------------------------------------------------------------
# exact index-set probe
# ---------------------------------------------------------------------------------------

def digits16(j, n=5):
    return [(j >> (4 * d)) & 15 for d in range(n)]


def probe_inputs(T, Hq, Hkv, D, rows, cols, seq, sign):
    """K and V of position j (stored in row j % rows) spell j in base 16 over dims 0..4;
    q has +-16^d there, so q.K_j = +-j exactly.  Every store cell is written once per
    column from the largest position each segment needs that maps to it."""
    q = torch.zeros((T, Hq, D), dtype=torch.bfloat16)
    for d in range(5):
        q[:, :, d] = sign * float(16 ** d)
    k = torch.zeros((rows, cols, Hkv, D), dtype=torch.bfloat16)
    for (qs, ql, col, ke) in seq:
        if ql <= 0:
            continue  # sees nothing; must not overwrite another segment's column
        for j in range(max(0, ke - rows), ke):
            k[j % rows, col, :, :5] = torch.tensor(digits16(j), dtype=torch.bfloat16)
    return q, k, k.clone()


def test_index_probe_decodes_interval_ends():
    T, Hq, Hkv, D, rows, cols = 24, 4, 2, 8, 11, 3
    seq = [(0, 5, 0, 30), (6, 4, 2, 3), (12, 7, 1, 17), (20, 0, 0, 5)]
    for causal, W in [(True, 0), (True, 6), (False, 0), (False, 9)]:
        good_seq = [s for s in seq if O.segment_status(s, T, rows, cols, W) == 0]
        seg_id, lo, hi, _ = O.visible_interval(np.array(seq), T, causal, W, rows, cols)
        for sign in (+1, -1):
            q, k, v = probe_inputs(T, Hq, Hkv, D, rows, cols, good_seq, sign)
            out, _, _ = O.sdpa_varlen(q, k, v, np.array(seq), causal, W, 64.0)
            dec = np.rint(out[:, :, :5]).astype(np.int64)
            val = sum(dec[:, :, d] * 16 ** d for d in range(5))
            for t in range(T):
                if seg_id[t] < 0 or hi[t] <= lo[t]:
                    assert np.all(out[t] == 0)
                    continue
                want = hi[t] - 1 if sign > 0 else lo[t]
                assert np.all(val[t] == want), (causal, W, t, val[t], lo[t], hi[t])
                # and against the brute-force predicate
                qs, ql, col, ke = seq[seg_id[t]]
                p = ke - ql + (t - qs)
                vis = [j for j in range(ke) if _visible(j, p, ke, causal, W)]
                assert want == (max(vis) if sign > 0 else min(vis))


# ---------------------------------------------------------------------------------------
# planted mistakes are caught (mutations of the oracle, on the CPU)
# ---------------------------------------------------------------------------------------

def _grid_disagrees(monkeypatch_ctx=None):
    rng = np.random.default_rng(77)
    for trial in range(30):
        causal = bool(trial % 2)
        W = [0, 2, 3][trial % 3]
        rows = 6
        segs, q, K, V = _rand_case(rng, T=8, Hq=4, Hkv=2, D=3, rows=rows, cols=2, S=2,
                                   max_q=3, max_kv=9, allow_bad=False)
        out, seg_id, status = O.sdpa_varlen(q, K, V, np.array(segs), causal, W, 0.9)
        ref, owners, ref_status = brute_force(q.tolist(), K.tolist(), V.tolist(), segs, causal, W, 0.9)
        if status != ref_status:
            return True
        for t in range(8):
            if seg_id[t] >= 0 and not np.allclose(out[t], ref[t], rtol=1e-12, atol=1e-12):
                return True
    return False


def test_grid_passes_unmutated():
    assert not _grid_disagrees()


def test_planted_window_off_by_one_is_caught(monkeypatch):
    def bad(i, q_len, kv_end, causal, window):
        p = kv_end - q_len + i
        hi = min(p + 1, kv_end) if causal else kv_end
        lo = max(0, p - window) if window > 0 else 0
        return lo, hi
    monkeypatch.setattr(O, "row_interval", bad)
    assert _grid_disagrees()


def test_planted_head_map_is_caught(monkeypatch):
    monkeypatch.setattr(O, "kv_head", lambda h, group: h % 2)
    assert _grid_disagrees()


def test_planted_ring_index_is_caught(monkeypatch):
    monkeypatch.setattr(O, "store_row", lambda j, rows: (j + 1) % rows)
    assert _grid_disagrees()


def test_planted_causal_drop_is_caught(monkeypatch):
    real = O.row_interval
    monkeypatch.setattr(O, "row_interval", lambda i, ql, ke, c, w: real(i, ql, ke, False, w))
    assert _grid_disagrees()


def test_overlapping_segments_make_all_their_rows_unspecified():
    q = np.ones((8, 1, 2))
    k = np.zeros((4, 2, 1, 2))
    v = np.ones((4, 2, 1, 2))
    seq = np.array([[0, 3, 0, 3], [2, 2, 1, 2], [5, 2, 0, 2]])  # first two share row 2
    out, seg_id, status = O.sdpa_varlen(q, k, v, seq, True, 0, 1.0)
    assert status == O.SEG_OVERLAP
    assert list(seg_id) == [-2, -2, -2, -2, -1, 2, 2, -1]
    assert np.all(out[5:7] == 1.0) and np.all(out[4] == 0) and np.all(out[7] == 0)
