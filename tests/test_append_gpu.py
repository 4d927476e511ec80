"""GPU parity of the KV append + attend entry (sdpa_varlen_append) against the oracle.

The stores after the call must equal the oracle's appended stores bit for bit (pure data
movement); the attention output must match the oracle's attention over those stores within
the usual tolerance, through every route."""

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


def _new_rows(call, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (call.T, call.Hkv, call.D)
    return (torch.randn(shape, generator=g).to(torch.bfloat16), torch.randn(shape, generator=g).to(torch.bfloat16))


def check_append(call, dev, seed, tag, k_new=None, v_new=None, seq=None):
    seq = call.seq_info if seq is None else seq
    if k_new is None:
        k_new, v_new = _new_rows(call, seed)
    k_ref, v_ref = O.kv_append(call.k_store, call.v_store, k_new, v_new, seq, call.window)
    k, v = call.k_store.to(dev), call.v_store.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.full((pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(seq)),), 255,
                    dtype=torch.uint8, device=dev)
    got = pkg.sdpa_varlen_append(call.q.to(dev), k_new.to(dev), v_new.to(dev), k, v,
                                 torch.from_numpy(np.ascontiguousarray(seq, dtype=np.int32)).to(dev),
                                 causal=call.causal, window=call.window, scale=call.scale,
                                 workspace=ws, status=status)
    torch.cuda.synchronize()
    assert torch.equal(k.cpu().view(torch.int16), k_ref.view(torch.int16)), f"{tag}: k_store differs"
    assert torch.equal(v.cpu().view(torch.int16), v_ref.view(torch.int16)), f"{tag}: v_store differs"
    ref, seg_id, st = O.sdpa_varlen(call.q, k_ref, v_ref, seq, call.causal, call.window, call.scale)
    _, lo, hi, _ = O.visible_interval(seq, call.T, call.causal, call.window, call.rows, call.cols)
    assert int(status.item()) == st, f"{tag}: status {int(status.item())} != {st}"
    assert_matches(got, ref, seg_id, lo, hi, tag=tag)


def test_append_decode_step(dev, route):
    # the batched decode step: each sequence's new row goes to position kv_end - 1
    check_append(synth.batched_decode(seed=1, S=32, rows=2048).calls[0], dev, 3, "decode")


def test_append_ring_window_segments(dev, route):
    wl = synth.mixed_step(seed=2)
    check_append(wl.calls[0], dev, 4, "ring")   # causal W=4096 segments on a 4111-row ring
    check_append(wl.calls[1], dev, 5, "draft")  # non-causal 16-row blocks on a flat store


def test_append_prefill_segment(dev, route):
    check_append(synth.long_causal_prefill(64, 512, 4096, seed=3).calls[0], dev, 6, "prefill")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_append_random_tables_with_invalid_and_overlapping_segments(dev, route, D):
    rng = np.random.default_rng(D + 7)
    for trial, (Hq, Hkv) in enumerate([(4, 1), (8, 2), (6, 3)]):
        call = synth.random_call(rng, D=D, Hq=Hq, Hkv=Hkv, T=90, S=7, rows=int(rng.choice([40, 300])),
                                 cols=8, causal=bool(trial % 2), window=int(rng.choice([0, 9])),
                                 max_q=20, max_kv=300, gen_seed=trial + D, distinct_cols=True)
        seq = np.array(call.seq_info, copy=True)
        seq[1, 1] = seq[0, 1] + 3                 # segment 1 may now overlap segment 0
        seq[2, 2] = call.cols + 4                 # column out of range
        check_append(call, dev, trial, f"D{D} trial{trial}", seq=seq)


def test_append_strided_new_rows(dev, route):
    call = synth.batched_decode(seed=4, S=16, rows=1024).calls[0]
    big_k, big_v = _new_rows(synth.batched_decode(seed=4, S=48, rows=1024).calls[0], 9)
    wide_k = torch.cat([big_k, big_k], dim=1)[: call.T]   # row stride 2 * Hkv * D
    wide_v = torch.cat([big_v, big_v], dim=1)[: call.T]
    k_new, v_new = wide_k[:, : call.Hkv], wide_v[:, : call.Hkv]
    assert not k_new.is_contiguous()
    check_append(call, dev, 0, "strided", k_new=k_new, v_new=v_new)


def test_append_in_a_captured_graph(dev):
    call = synth.batched_decode(seed=5, S=8, rows=512).calls[0]
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    seq = torch.from_numpy(call.seq_info).to(dev)
    kn = torch.empty((call.T, call.Hkv, call.D), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    out = torch.empty((call.T, call.Hq, call.D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkg.workspace_bytes(call.T, call.Hq, call.Hkv, call.D, len(call.seq_info)),
                     dtype=torch.uint8, device=dev)
    kw = dict(causal=True, scale=call.scale, out=out, workspace=ws)
    pkg.sdpa_varlen_append(q, kn, vn, k, v, seq, **kw)  # warm
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.sdpa_varlen_append(q, kn, vn, k, v, seq, **kw)
    k_ref, v_ref = call.k_store, call.v_store
    for step in range(3):
        a, b = _new_rows(call, 100 + step)
        kn.copy_(a)
        vn.copy_(b)
        g.replay()
        torch.cuda.synchronize()
        k_ref, v_ref = O.kv_append(k_ref, v_ref, a, b, call.seq_info, 0)
        assert torch.equal(k.cpu().view(torch.int16), k_ref.view(torch.int16))
        ref, seg_id, _ = O.sdpa_varlen(call.q, k_ref, v_ref, call.seq_info, True, 0, call.scale)
        _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, True, 0, call.rows, call.cols)
        assert_matches(out, ref, seg_id, lo, hi, tag=f"graph step {step}")


@pytest.mark.parametrize("rows,n,src,dst", [(64, 40, 1, 3), (64, 64, 0, 2), (64, 200, 2, 0), (512, 0, 1, 2),
                                             (300, 123, 3, 3)])
def test_seq_clone_matches_the_oracle_bit_for_bit(dev, rows, n, src, dst):
    g = torch.Generator().manual_seed(rows + n)
    k0 = torch.randn(rows, 4, 2, 128, generator=g).to(torch.bfloat16)
    v0 = torch.randn(rows, 4, 2, 128, generator=g).to(torch.bfloat16)
    k, v = k0.to(dev), v0.to(dev)
    pkg.sdpa_seq_clone(k, v, src, dst, n)
    torch.cuda.synchronize()
    k_ref, v_ref = O.seq_clone(k0, v0, src, dst, n)
    assert torch.equal(k.cpu().view(torch.int16), k_ref.view(torch.int16))
    assert torch.equal(v.cpu().view(torch.int16), v_ref.view(torch.int16))


def test_cloned_sequence_attends_bit_identically(dev, route):
    # the mixed step's ring segments, each cloned into a fresh column: same outputs, bit for bit
    call = synth.mixed_step(seed=3).calls[0]
    k, v = call.k_store.to(dev), call.v_store.to(dev)
    seq = np.array(call.seq_info, copy=True)
    free = call.cols - 1  # the scratch column
    for s in range(len(seq)):
        q_start, q_len, col, kv_end = (int(x) for x in seq[s])
        one = np.array([[q_start, q_len, col, kv_end]], dtype=np.int32)
        a = pkg.sdpa_varlen(call.q.to(dev), k, v, torch.from_numpy(one).to(dev), causal=True,
                            window=call.window, scale=call.scale)
        pkg.sdpa_seq_clone(k, v, col, free, kv_end)
        one[0, 2] = free
        b = pkg.sdpa_varlen(call.q.to(dev), k, v, torch.from_numpy(one).to(dev), causal=True,
                            window=call.window, scale=call.scale)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), s
