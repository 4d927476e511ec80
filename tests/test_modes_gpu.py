"""GPU parity of the per-segment mask mode (sdpa_varlen_modes) against the oracle.

Causal sliding-window target segments and non-causal draft blocks share one store and one
launch (the per-model `causal` of the "[executorch][cuda] Add a length-aware Triton SDPA over
per-sequence KV columns" stack, moved into the segment table).  Each case runs on every
route; a uniform table must give the call-level entry's output bit for bit."""

import numpy as np
import pytest
import torch

import varlen_gqa_attention_gb300 as pkg
from oracle import sdpa_varlen_oracle as O
from workloads import synth

from parity import assert_matches

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


def _i32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def run_modes(call, modes, dev, seq=None, k=None, v=None, status=None):
    seq = call.seq_info if seq is None else seq
    ws = torch.full((pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(seq)),), 255,
                    dtype=torch.uint8, device=dev)
    return pkg.sdpa_varlen_modes(call.q.to(dev), call.k_store.to(dev) if k is None else k,
                                 call.v_store.to(dev) if v is None else v, _i32(seq, dev),
                                 _i32(modes, dev), scale=call.scale, workspace=ws, status=status)


def check_modes(call, modes, dev, tag, seq=None, k=None, v=None):
    seq = call.seq_info if seq is None else seq
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = run_modes(call, modes, dev, seq=seq, k=None if k is None else k.to(dev),
                    v=None if v is None else v.to(dev), status=status)
    torch.cuda.synchronize()
    kk = call.k_store if k is None else k
    vv = call.v_store if v is None else v
    ref, seg_id, st = O.sdpa_varlen(call.q, kk, vv, seq, True, 0, call.scale, seg_mode=modes)
    _, lo, hi, _ = O.visible_interval(seq, call.T, True, 0, call.rows, call.cols, seg_mode=modes)
    assert int(status.item()) == st, f"{tag}: status {int(status.item())} != {st}"
    return assert_matches(got, ref, seg_id, lo, hi, tag=tag)


def shared_store_step(seed=0, **kw):
    """The one-store mixed step: causal W=4096 targets and non-causal draft blocks."""
    call = synth.mixed_step_one_store(seed=seed, **kw).calls[0]
    return call, call.seg_mode


def poison_invisible_modes(call, modes, value=float("nan")):
    """Store copies with every cell that no valid segment sees under its own mode set to value."""
    k, v = call.k_store.clone(), call.v_store.clone()
    needed = np.zeros((call.rows, call.cols), dtype=bool)
    for seg, (_, w) in zip(np.asarray(call.seq_info, dtype=np.int64), np.asarray(modes, dtype=np.int64)):
        w = int(w)
        if O.segment_status(seg, call.T, call.rows, call.cols, w):
            continue
        _, q_len, col, kv_end = (int(x) for x in seg)
        span = O.needed_span(q_len, kv_end, w)
        for j in range(kv_end - span, kv_end):
            needed[j % call.rows, col] = True
    mask = torch.from_numpy(~needed)
    k[mask] = value
    v[mask] = value
    return k, v


def test_target_and_draft_segments_in_one_launch(dev, route):
    call, modes = shared_store_step(seed=1)
    check_modes(call, modes, dev, "shared store")


def test_cells_outside_each_segments_own_mask_are_never_read(dev, route):
    call, modes = shared_store_step(seed=2, n_target=5, n_draft=6)
    k, v = poison_invisible_modes(call, modes)
    check_modes(call, modes, dev, "poisoned", k=k, v=v)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_random_tables_with_random_modes(dev, route, D):
    rng = np.random.default_rng(D + 31)
    for trial, (Hq, Hkv) in enumerate([(4, 1), (8, 2), (6, 3)]):
        call = synth.random_call(rng, D=D, Hq=Hq, Hkv=Hkv, T=120, S=9, rows=int(rng.choice([48, 400])),
                                 cols=6, causal=True, window=0, max_q=24, max_kv=420,
                                 gen_seed=trial + 3 * D)
        modes = np.stack([rng.integers(0, 2, size=9), rng.choice([0, -3, 1, 5, 17, 64], size=9)], 1)
        check_modes(call, modes.astype(np.int32), dev, f"D{D} trial{trial}")


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 37), (False, 9)])
def test_a_uniform_table_equals_the_call_level_entry_bit_for_bit(dev, route, causal, window):
    call = synth.random_call(np.random.default_rng(window + 2 * causal), D=128, Hq=8, Hkv=2, T=150,
                             S=10, rows=512, cols=10, causal=causal, window=window, max_q=30,
                             max_kv=500, gen_seed=5, distinct_cols=True)
    modes = np.array([[int(causal), window]] * len(call.seq_info), dtype=np.int32)
    a = pkg.sdpa_varlen(call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev),
                        _i32(call.seq_info, dev), causal=causal, window=window, scale=call.scale)
    b = run_modes(call, modes, dev)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_modes_change_between_graph_replays(dev):
    # the table is read on the device: one captured graph serves any mix of modes
    call, modes = shared_store_step(seed=3, n_target=4, n_draft=4, Hq=16, Hkv=4, T=128)
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    seq, md = _i32(call.seq_info, dev), _i32(modes, dev)
    out = torch.empty((call.T, call.Hq, call.D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(call.seq_info)),
                     dtype=torch.uint8, device=dev)
    kw = dict(scale=call.scale, out=out, workspace=ws)
    pkg.sdpa_varlen_modes(q, k, v, seq, md, **kw)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.sdpa_varlen_modes(q, k, v, seq, md, **kw)
    rng = np.random.default_rng(7)
    for step in range(3):
        m = modes.copy()
        m[:, 0] = rng.integers(0, 2, size=len(m))
        m[:4, 1] = rng.choice([call.rows - 15, 300, 1], size=4)  # target windows keep them valid
        md.copy_(_i32(m, dev))
        g.replay()
        torch.cuda.synchronize()
        ref, seg_id, _ = O.sdpa_varlen(call.q, call.k_store, call.v_store, call.seq_info, True, 0,
                                       call.scale, seg_mode=m)
        _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, True, 0, call.rows, call.cols, seg_mode=m)
        assert_matches(out, ref, seg_id, lo, hi, tag=f"replay {step}")
