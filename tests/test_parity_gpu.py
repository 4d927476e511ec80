"""GPU parity: the CUDA library (through the C interface) against the CPU oracle.

Every test runs on cuda:0 and compares element by element with the fp64 oracle on the same
seeded inputs (tolerances in tests/parity.py).  Both kernels are checked on every case by
forcing each route (the auto route sends long segments to the prefill kernel).
"""

import numpy as np
import pytest
import torch

import varlen_gqa_attention_gb300 as pkg
from oracle import sdpa_varlen_oracle as O
from workloads import synth

from parity import (assert_matches, check_call, decode_probe, oracle, poison_invisible, probe_call,
                    run_call)

pytestmark = pytest.mark.gpu

ROUTES = [pkg.ROUTE_AUTO, pkg.ROUTE_SPLITK, pkg.ROUTE_PREFILL]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(params=ROUTES, ids=["auto", "splitk", "prefill"])
def route(request):
    pkg.set_route_policy(request.param)
    yield request.param
    pkg.set_route_policy(pkg.ROUTE_AUTO)


def test_native_library_is_loaded(dev):
    lib = pkg.library()
    import varlen_gqa_attention_gb300._build as b
    maps = open("/proc/self/maps").read()
    assert b.lib_path() in maps
    assert lib.sdpa_version() == 100


def test_tiny_causal_prefill(dev, route):
    call = synth.tiny_causal_prefill(seed=0).calls[0]
    check_call(call, dev, tag="tiny")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_d64_long_prefill_full(dev, route, seed):
    call = synth.long_causal_prefill(64, 512, 16384, seed=seed).calls[0]
    check_call(call, dev, tag=f"d64 seed {seed}")


def test_d128_long_prefill_sampled_rows(dev, route):
    call = synth.long_causal_prefill(128, 4096, 131072, seed=0).calls[0]
    # both ends, both sides of every 256-query-row boundary (units hold 32 query rows at group
    # 8, key tiles 128 positions), and random rows in between
    edges = [b + d for b in range(0, 4097, 256) for d in (-1, 0) if 0 <= b + d < 4096]
    rows = sorted(set([0, 1, 15, 16, 17, 31, 32, 127, 128, 2047, 2048, 4094, 4095] + edges +
                      list(np.random.default_rng(0).integers(0, 4096, 40))))
    check_call(call, dev, rows_subset=rows, tag="d128 sampled")


def test_d128_prefill_full_over_several_units(dev, route):
    # every row of a 768 x 6000 causal prefill (24 units of 256 packed rows, ragged last
    # key tile)
    call = synth.long_causal_prefill(128, 768, 6000, seed=4).calls[0]
    check_call(call, dev, tag="d128 768x6000")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_windowed_prefill_whose_keys_wrap_the_ring(dev, route, D):
    """Long sliding-window chunks on a ring store of window + q_len - 1 rows whose keys cross
    the ring's end (the prefill kernel tiles them in two parts at the wrap)."""
    W, q_len, Hq, Hkv = 300, 64, 8, 2
    rows, cols = W + q_len - 1, 4
    segs = [(0, q_len, 0, 2000), (q_len, q_len, 1, 363 * 3 + 40), (2 * q_len, 40, 2, 1700), (2 * q_len + 40, 1, 3, 900)]
    g = torch.Generator().manual_seed(D)
    T = 2 * q_len + 41
    call = synth.Call(T, Hq, Hkv, D, rows, cols, np.array(segs, dtype=np.int32), True, W, D ** -0.5,
                      torch.randn((T, Hq, D), generator=g).to(torch.bfloat16),
                      torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16),
                      torch.randn((rows, cols, Hkv, D), generator=g).to(torch.bfloat16))
    for qs, ql, col, ke in segs[:3]:
        first = ke - min(ke, ql + W - 1)
        assert first // rows != (ke - 1) // rows  # the keys wrap
    check_call(call, dev, tag=f"ring wrap D={D}")


def test_ring_window_prefill_workload_sampled_rows(dev, route):
    call = synth.ring_window_prefill(seed=0).calls[0]
    rows = sorted(set([0, 1, 15, 16, 31, 32, 1023, 1024, 2046, 2047] +
                      list(np.random.default_rng(1).integers(0, call.T, 24))))
    check_call(call, dev, rows_subset=rows, tag="ring prefill")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_batched_decode_full(dev, route, seed):
    call = synth.batched_decode(seed=seed).calls[0]
    check_call(call, dev, tag=f"decode seed {seed}")


@pytest.mark.parametrize("seed", [0, 1])
def test_mixed_step_full(dev, route, seed):
    wl = synth.mixed_step(seed=seed)
    T = wl.calls[-1].row_end
    out = torch.full((T, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    for c in wl.calls:
        run_call(c, dev, out=out[c.row_begin:c.row_end])  # each call owns its half
    torch.cuda.synchronize()
    for c in wl.calls:
        ref, seg_id, _ = oracle(c)
        _, lo, hi, _ = O.visible_interval(c.seq_info, c.T, c.causal, c.window, c.rows, c.cols)
        assert_matches(out[c.row_begin:c.row_end], ref, seg_id, lo, hi, tag=f"mixed causal={c.causal}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 5), (False, 7), (True, 1)])
def test_random_tables(dev, route, D, causal, window):
    rng = np.random.default_rng(D * 100 + window * 3 + int(causal))
    for trial, (Hq, Hkv) in enumerate([(4, 1), (8, 2), (6, 3), (16, 16)]):
        rows = int(rng.choice([40, 97, 300]))
        call = synth.random_call(rng, D=D, Hq=Hq, Hkv=Hkv, T=80, S=6, rows=rows, cols=3,
                                 causal=causal, window=window, max_q=24, max_kv=320,
                                 gen_seed=trial + 10 * D)
        check_call(call, dev, tag=f"D{D} Hq{Hq}/{Hkv} {causal} W{window} rows{rows}")


def test_ring_store_long_window(dev, route):
    # causal window 300 on a 315-row ring (window + max_write - 1), long positions
    rng = np.random.default_rng(5)
    call = synth.random_call(rng, D=128, Hq=8, Hkv=2, T=64, S=4, rows=315, cols=5, causal=True,
                             window=300, max_q=16, max_kv=5000, gen_seed=3)
    check_call(call, dev, tag="ring")


def test_invalid_segments_set_status_and_zero_rows(dev, route):
    call = synth.random_call(np.random.default_rng(9), D=64, Hq=4, Hkv=2, T=40, S=2, rows=64, cols=2,
                             causal=True, window=0, max_q=8, max_kv=60, gen_seed=4, allow_gaps=False)
    bad = np.array([[0, 5, 0, 20],      # valid
                    [5, 3, 2, 10],      # bad column
                    [8, -1, 0, 3],      # negative q_len
                    [9, 4, 1, 65],      # kv_end beyond the 64 rows, no window
                    [13, 4, 1, -2],     # negative kv_end
                    [17, 30, 0, 10],    # q range beyond T
                    [20, 3, 1, 12],     # valid
                    [22, 2, 0, 5]],     # overlaps the previous one
                   dtype=np.int32)
    call.seq_info = bad
    check_call(call, dev, tag="invalid")


def test_workspace_status_reads_back_the_calls_status_bits(dev, route):
    """Without status_dev, the status of the last call is read back from its workspace."""
    call = synth.random_call(np.random.default_rng(9), D=64, Hq=4, Hkv=2, T=40, S=2, rows=64, cols=2,
                             causal=True, window=0, max_q=8, max_kv=60, gen_seed=4, allow_gaps=False)
    tables = [np.array([[0, 5, 0, 20], [5, 3, 2, 10], [9, 4, 1, 65], [20, 3, 1, 12], [22, 2, 0, 5]],
                       dtype=np.int32),
              np.array([[0, 5, 0, 20], [20, 3, 1, 12]], dtype=np.int32)]
    ws = torch.full((pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, 5),), 255, dtype=torch.uint8,
                    device=dev)
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    for tab in tables:
        seq = torch.from_numpy(tab).to(dev)
        pkg.sdpa_varlen(q, k, v, seq, causal=True, scale=call.scale, workspace=ws)
        _, _, _, st = O.visible_interval(tab, call.T, True, 0, call.rows, call.cols)
        assert pkg.workspace_status(ws) == st  # the second table is clean: 0


def test_nan_in_invisible_cells_changes_no_output_bit(dev, route):
    wl = synth.batched_decode(seed=1, S=8, rows=2048)
    call = wl.calls[0]
    clean = run_call(call, dev).clone()
    k, v = poison_invisible(call)
    dirty = run_call(call, dev, k=k.to(dev), v=v.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(clean.view(torch.int16), dirty.view(torch.int16))
    rng = np.random.default_rng(3)
    call = synth.random_call(rng, D=128, Hq=8, Hkv=2, T=64, S=4, rows=200, cols=5, causal=True,
                             window=60, max_q=16, max_kv=900, gen_seed=3)
    clean = run_call(call, dev).clone()
    k, v = poison_invisible(call)
    dirty = run_call(call, dev, k=k.to(dev), v=v.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(clean.view(torch.int16), dirty.view(torch.int16))


@pytest.mark.parametrize("causal,window,rows", [(True, 0, 5000), (True, 37, 52), (False, 0, 5000),
                                                (False, 23, 40), (True, 200, 215)])
def test_index_sets_are_bit_exact(dev, route, causal, window, rows):
    rng = np.random.default_rng(rows + window)
    max_q = min(40, rows - window + 1) if window else 40
    # each segment owns its column, so every store cell spells one position
    call = synth.random_call(rng, D=64, Hq=8, Hkv=2, T=200, S=8, rows=rows, cols=8, causal=causal,
                             window=window, max_q=max_q, max_kv=min(4000, 3 * rows), gen_seed=1,
                             distinct_cols=True)
    call.scale = 64.0
    seg_id, lo, hi, _ = O.visible_interval(call.seq_info, call.T, causal, window, rows, call.cols)
    for sign in (+1, -1):
        q, k = probe_call(call, sign)
        out = run_call(call, dev, q=q.to(dev), k=k.to(dev), v=k.to(dev))
        torch.cuda.synchronize()
        got = decode_probe(out)
        for t in range(call.T):
            if seg_id[t] == O.UNCOVERED or (seg_id[t] >= 0 and hi[t] <= lo[t]):
                assert bool((out[t].view(torch.int16) == 0).all()), t
            elif seg_id[t] >= 0:
                want = hi[t] - 1 if sign > 0 else lo[t]
                assert np.all(got[t] == want), (t, sign, got[t], lo[t], hi[t])


def test_graph_replay_with_new_lengths(dev, route):
    T, Hq, Hkv, D, rows, cols, S = 64, 8, 2, 128, 1024, 5, 4
    rng = np.random.default_rng(11)
    base = synth.random_call(rng, D=D, Hq=Hq, Hkv=Hkv, T=T, S=S, rows=rows, cols=cols, causal=True,
                             window=0, max_q=16, max_kv=rows, gen_seed=5)
    q, k, v = base.q.to(dev), base.k_store.to(dev), base.v_store.to(dev)
    seq = torch.zeros((S, 4), dtype=torch.int32, device=dev)
    out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkg.workspace_bytes(T, Hq, Hkv, D, S), dtype=torch.uint8, device=dev)
    seq.copy_(torch.from_numpy(base.seq_info))
    pkg.sdpa_varlen(q, k, v, seq, causal=True, scale=base.scale, out=out, workspace=ws)  # warm
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.sdpa_varlen(q, k, v, seq, causal=True, scale=base.scale, out=out, workspace=ws)
    tables = [
        np.array([[0, 16, 0, 1000], [16, 1, 1, 5], [20, 9, 2, 9], [40, 3, 4, 3]]),
        np.array([[3, 1, 3, 1], [4, 0, 0, 0], [10, 16, 1, 700], [30, 12, 0, 12]]),
        np.array([[0, 8, 4, 1024], [8, 8, 3, 512], [16, 8, 2, 256], [24, 8, 1, 8]]),
    ]
    for tab in tables:
        seq.copy_(torch.from_numpy(tab.astype(np.int32)))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, seg_id, _ = O.sdpa_varlen(base.q, base.k_store, base.v_store, tab, True, 0, base.scale)
        _, lo, hi, _ = O.visible_interval(tab, T, True, 0, rows, cols)
        assert_matches(out, ref, seg_id, lo, hi, tag=f"replay {tab[:, 1]}")


def test_dense_entry_equals_one_segment_call(dev):
    call = synth.long_causal_prefill(128, 300, 2000, seed=2).calls[0]
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    a = pkg.sdpa_causal_prefill(q, k[:, 0].contiguous(), v[:, 0].contiguous(), call.scale)
    b = run_call(call, dev, q=q, k=k, v=v)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = O.sdpa_causal_prefill(call.q, call.k_store[:, 0], call.v_store[:, 0], call.scale)
    err = np.abs(a.double().cpu().numpy() - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_strided_q_and_out(dev, route):
    call = synth.random_call(np.random.default_rng(4), D=128, Hq=8, Hkv=4, T=48, S=3, rows=256,
                             cols=3, causal=True, window=0, max_q=16, max_kv=256, gen_seed=8)
    big = torch.zeros((48, 8, 3 * 128), dtype=torch.bfloat16, device=dev)
    big[:, :, 128:256] = call.q.to(dev)
    q = big[:, :, 128:256]
    ob = torch.zeros((48, 10, 128), dtype=torch.bfloat16, device=dev)
    out = ob[:, 1:9]
    run_call(call, dev, q=q, out=out)
    torch.cuda.synchronize()
    ref, seg_id, _ = oracle(call)
    _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, True, 0, call.rows, call.cols)
    assert_matches(out, ref, seg_id, lo, hi, tag="strided")
    assert bool((ob[:, 0].view(torch.int16) == 0).all()) and bool((ob[:, 9].view(torch.int16) == 0).all())


def test_empty_step_and_zero_segments(dev):
    call = synth.random_call(np.random.default_rng(1), D=64, Hq=4, Hkv=1, T=16, S=1, rows=32, cols=1,
                             causal=True, window=0, max_q=4, max_kv=32, gen_seed=1)
    call.seq_info = np.zeros((0, 4), dtype=np.int32)
    out = run_call(call, dev)
    torch.cuda.synchronize()
    assert bool((out.view(torch.int16) == 0).all())


@pytest.mark.parametrize("D", [64, 128, 256])
def test_short_pieces_are_deterministic_and_exact(dev, route, D):
    # one 16-query segment per KV head: every CTA gets one or two short pieces of different
    # units, the case where an epilogue could read O before its last PV landed
    call = synth.random_call(np.random.default_rng(D), D=D, Hq=32, Hkv=8, T=64, S=1, rows=8192, cols=2,
                             causal=False, window=0, max_q=1, max_kv=1, gen_seed=D, allow_gaps=False)
    call.seq_info = np.array([[0, 16, 1, 5186]], dtype=np.int32)
    outs = [run_call(call, dev).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))
    ref, seg_id, _ = oracle(call)
    _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, False, 0, call.rows, call.cols)
    assert_matches(outs[0], ref, seg_id, lo, hi, tag=f"short pieces D{D}")


def test_segment_table_larger_than_the_scheduler_cache(dev, route):
    # 1500 segments: more than the scheduler stages in shared memory, so it walks the
    # workspace copy of the table instead
    rng = np.random.default_rng(1500)
    call = synth.random_call(rng, D=64, Hq=4, Hkv=2, T=3000, S=1500, rows=64, cols=8, causal=True,
                             window=0, max_q=2, max_kv=48, gen_seed=77)
    check_call(call, dev, tag="S=1500")


@pytest.mark.parametrize("Hq,Hkv", [(32, 1), (128, 1), (24, 8)])
def test_large_and_odd_head_groups(dev, route, Hq, Hkv):
    # group 32 and 128 fill a 128-row prefill tile with 4 and 1 query rows; group 3 does not
    # divide 128 and always takes the split-K kernel
    rng = np.random.default_rng(Hq * 7 + Hkv)
    call = synth.random_call(rng, D=64, Hq=Hq, Hkv=Hkv, T=40, S=4, rows=300, cols=2, causal=True,
                             window=0, max_q=12, max_kv=300, gen_seed=Hq + Hkv)
    check_call(call, dev, tag=f"Hq{Hq}/Hkv{Hkv}")


@pytest.mark.parametrize("T,Hq,Hkv,segs", [
    # more packed rows than the scheduler's shared-memory owner map, and more units
    (9000, 16, 2, [(0, 4000, 0, 4000), (4000, 3000, 1, 7000), (7000, 2000, 2, 9500)]),
    # rows within the owner map, units beyond the shared-memory unit table
    (8000, 32, 4, [(0, 5000, 0, 5000), (5000, 2990, 2, 8000)]),
])
def test_more_rows_and_units_than_the_scheduler_stages(dev, route, T, Hq, Hkv, segs):
    D, rows, cols = 64, 10000, 3
    g = torch.Generator().manual_seed(T + Hq)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    call = synth.Call(T, Hq, Hkv, D, rows, cols, np.array(segs, dtype=np.int32), True, 0,
                      1.0 / np.sqrt(D), q, k, v)
    rng = np.random.default_rng(T)
    sample = set(rng.choice(T, size=120, replace=False).tolist())
    for (qs, ql, _, _) in segs:  # segment edges and the uncovered tail
        sample.update([qs, qs + ql - 1])
    sample.update(range(T - 12, T))
    check_call(call, dev, rows_subset=sorted(sample), tag=f"T={T}")


def _table_call(S, Hq, Hkv, q_len, seed, edit=None):
    # S segments of q_len rows (an int, or a cycle of lengths), packed in order with a 5-row
    # uncovered tail, over a 1024-row store (one column each); `edit` may rewrite the table
    D, rows, cols = 64, 1024, S + 1
    rng = np.random.default_rng(seed)
    lens = [q_len] * S if isinstance(q_len, int) else [q_len[s % len(q_len)] for s in range(S)]
    starts = np.concatenate([[0], np.cumsum(lens)]).tolist()
    segs = [[starts[s], lens[s], s, int(rng.integers(lens[s], rows + 1))] for s in range(S)]
    if edit is not None:
        edit(segs, cols)
    T = starts[S] + 5
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    return synth.Call(T, Hq, Hkv, D, rows, cols, np.array(segs, dtype=np.int32), True, 0,
                      1.0 / np.sqrt(D), q, k, v)


def _messy(segs, cols):
    segs[4][0] = segs[3][0] + 1   # 3 and 4 share rows: both dropped
    segs[7][2] = cols             # column out of range
    segs[9][1] = 0                # empty
    segs[11][3] = -1              # negative kv_end
    segs[20][0] = segs[31][0]     # 20 and 31 share rows, far apart in the table


def _reversed(segs, cols):
    segs.reverse()                # disjoint rows, but not in row order


@pytest.mark.parametrize("S,Hq,Hkv,q_len,edit", [
    (32, 32, 8, 16, None),     # 32 segments, 512 split-K units: the shortest chains
    (32, 32, 8, 17, None),     # 32 segments, 768 units: unit steps over ranges per thread
    (33, 16, 2, 1, None),      # 33 segments, 66 units: block-wide segment steps, one unit per thread
    (32, 16, 2, 3, _messy),    # invalid, empty and overlapping segments in the one-warp steps
    (40, 16, 2, 3, _messy),    # the same table shape through the block-wide steps
    (32, 16, 2, 3, _reversed),  # disjoint segments out of row order: the pairwise overlap test
    (20, 32, 8, (40, 3), None),  # 80 prefill and 80 split-K units (auto route) in one block
], ids=["s32_u512", "s32_u768", "s33_u66", "s32_messy", "s40_messy", "s32_reversed", "s20_two_routes"])
def test_scheduler_paths_at_their_limits(dev, route, S, Hq, Hkv, q_len, edit):
    call = _table_call(S, Hq, Hkv, q_len, seed=S * 100 + int(np.sum(q_len)), edit=edit)
    check_call(call, dev, tag=f"S={S} q_len={q_len}")


def _equal_length_call(S, Hq, Hkv, q_len, kv_lo, kv_hi, seed, window=0):
    # S segments of q_len rows with kv_end in [kv_lo, kv_hi], one column each
    D, cols = 64, S + 1
    rows = kv_hi
    rng = np.random.default_rng(seed)
    segs = [[s * q_len, q_len, s, int(rng.integers(kv_lo, kv_hi + 1))] for s in range(S)]
    T = S * q_len
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(rows, cols, Hkv, D, generator=g).to(torch.bfloat16)
    return synth.Call(T, Hq, Hkv, D, rows, cols, np.array(segs, dtype=np.int32), True, window,
                      1.0 / np.sqrt(D), q, k, v)


@pytest.mark.parametrize("S,Hq,Hkv,q_len,kv_lo,kv_hi,window", [
    (19, 128, 16, 1, 2000, 2000, 0),     # 304 equal split-K units, one per CTA (small scheduler)
    (19, 128, 16, 1, 1950, 2000, 0),     # near-equal lengths: still whole units
    (37, 64, 8, 1, 1980, 2000, 0),       # 296 units through the block-wide scheduler
    (1, 16, 2, 2048, 8192, 8192, 1024),  # 128 windowed prefill units of one long segment
    (1, 16, 2, 2048, 8192, 8192, 0),     # the same without a window: long, uneven units split
], ids=["s19_equal", "s19_near_equal", "s37_general", "prefill_window", "prefill_no_window"])
def test_whole_unit_phases(dev, route, S, Hq, Hkv, q_len, kv_lo, kv_hi, window):
    # phases of short, even units give each CTA one whole unit (no partial slots)
    call = _equal_length_call(S, Hq, Hkv, q_len, kv_lo, kv_hi, seed=S + q_len + kv_lo, window=window)
    rows = None
    if call.T > 256:
        rng = np.random.default_rng(5)
        rows = sorted(set(rng.choice(call.T, size=160, replace=False).tolist()) | {0, call.T - 1})
    check_call(call, dev, rows_subset=rows, tag=f"S={S} q_len={q_len}")


def _multi_phase_prefill_call():
    # 8 prefill segments of 512 rows over 16384 keys each: 16 (segment, KV head) groups whose
    # units re-read 8 MB of K/V each, so the tile line is cut into several phases
    S, ql, kv, Hq, Hkv, D = 8, 512, 16384, 16, 2, 128
    g = torch.Generator().manual_seed(88)
    q = torch.randn(S * ql, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(kv, S, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(kv, S, Hkv, D, generator=g).to(torch.bfloat16)
    si = np.array([(s * ql, ql, s, kv) for s in range(S)], dtype=np.int32)
    return synth.Call(S * ql, Hq, Hkv, D, kv, S, si, True, 0, 1.0 / np.sqrt(D), q, k, v)


@pytest.mark.parametrize("which", ["draft_blocks", "prefill_groups"])
def test_multi_phase_calls_stay_inside_the_workspace(dev, route, which):
    # several phases add (unit, CTA) pairs; the partial slots must hold them all and no byte
    # past the workspace may change
    call = synth.mixed_step(seed=2).calls[1] if which == "draft_blocks" else _multi_phase_prefill_call()
    n = pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(call.seq_info))
    big = torch.full((n + (1 << 20),), 0xA5, dtype=torch.uint8, device=dev)
    ws = big[:n]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = pkg.sdpa_varlen(call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev),
                          torch.from_numpy(call.seq_info).to(dev), causal=call.causal, window=call.window,
                          scale=call.scale, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert bool((big[n:] == 0xA5).all()), "bytes past the workspace changed"
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(call.T, size=96, replace=False),
                                     call.seq_info[:, 0], call.seq_info[:, 0] + call.seq_info[:, 1] - 1]))
    ref, seg_id, st = oracle(call, rows_subset=rows)
    _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, call.causal, call.window, call.rows, call.cols)
    assert int(status.item()) == st
    assert_matches(got, ref, seg_id, lo, hi, rows=rows, tag=which)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_the_tensor_memory_prefill_kernel_is_usable(dev, D):
    # if its set-up failed (e.g. more shared memory than an SM has), every call would quietly
    # take the split-K kernel: same results, far slower
    assert pkg.prefill_available(D)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("q_len", [1, 2])
def test_few_long_decode_sequences_split_over_dozens_of_ctas(dev, D, q_len):
    # two sequences of 60000 and 30000 keys: each (sequence, KV head) unit is cut over tens
    # of CTAs, more slots than the last CTA can stage in shared memory, so its merge reads
    # them straight from L2
    rows, Hq, Hkv = 65536, 16, 2
    g = torch.Generator().manual_seed(D + q_len)
    T = 2 * q_len
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(rows, 3, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(rows, 3, Hkv, D, generator=g).to(torch.bfloat16)
    si = np.array([(0, q_len, 0, 60000), (q_len, q_len, 2, 30000)], dtype=np.int32)
    call = synth.Call(T, Hq, Hkv, D, rows, 3, si, True, 0, 1.0 / np.sqrt(D), q, k, v)
    check_call(call, dev, tag=f"long decode D{D} q_len{q_len}")
