"""The allocation-free entry point, sdpa_varlen_splitk_static.

Some callers cannot allocate device memory (a runtime with a fixed memory plan, a plugin
that must not call cudaMalloc, a binding with no device allocator), so they cannot hand
sdpa_varlen a workspace.  sdpa_varlen_splitk_static keeps its scratch in a static device
array of the library instead.  These tests call it through the C interface (ctypes, no
torch allocation on its path) and check it, twice in a row (the second call finds the first
call's leftovers in the shared array), element by element against the fp64 CPU oracle and
against sdpa_varlen on the same inputs.  One case is sized so that its scratch only fits
the array at one CTA per SM (the entry's reduced grid).  This file is collected last so that
a failure here cannot hide the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import varlen_gqa_attention_gb300 as pkg
from oracle import sdpa_varlen_oracle as O
from workloads import synth

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3  # the parity tolerance of the other GPU tests


def _fn():
    lib = pkg.library()
    f = lib.sdpa_varlen_splitk_static
    c_i64, c_int, c_vp, c_f = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    f.restype = c_int
    f.argtypes = [c_vp, c_i64, c_int, c_int, c_i64, c_i64, c_vp, c_vp, c_i64, c_int, c_int, c_vp,
                  c_int, c_int, c_int, c_f, c_vp, c_i64, c_i64, c_vp, c_vp]
    return lib, f


def _static_call(call, q, k, v, seq, out, status):
    lib, f = _fn()
    code = f(q.data_ptr(), call.T, call.Hq, call.D, q.stride(0), q.stride(1), k.data_ptr(), v.data_ptr(),
             call.rows, call.cols, call.Hkv, seq.data_ptr() if seq.numel() else None, seq.shape[0],
             int(call.causal), call.window, call.scale, out.data_ptr(), out.stride(0), out.stride(1),
             status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 0, lib.sdpa_last_error().decode()


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _fallback_case():
    """T=2048 packed rows in 8 segments of 256 queries, Hq=16, Hkv=2, D=128: on a 152-SM
    GB300 its scratch needs more than the array at two split-K CTAs per SM and fits at one
    (tests/test_host_arith.py checks those two sizes on the CPU)."""
    rng = np.random.default_rng(77)
    T, S, rows, cols = 2048, 8, 1024, 9
    segs = [(256 * s, 256, s, int(rng.integers(256, rows + 1))) for s in range(S)]
    g = torch.Generator().manual_seed(78)
    q = torch.randn((T, 16, 128), generator=g).to(torch.bfloat16)
    k = torch.randn((rows, cols, 2, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((rows, cols, 2, 128), generator=g).to(torch.bfloat16)
    return synth.Call(T, 16, 2, 128, rows, cols, np.array(segs, dtype=np.int32), True, 0, 128 ** -0.5, q, k, v)


def _cases():
    rng = np.random.default_rng(21)
    yield synth.batched_decode(seed=2).calls[0]
    yield synth.random_call(rng, D=128, Hq=16, Hkv=2, T=96, S=6, rows=1500, cols=7, causal=True, window=0,
                            max_q=20, max_kv=1500, gen_seed=5)
    yield synth.random_call(rng, D=64, Hq=8, Hkv=2, T=64, S=5, rows=300, cols=6, causal=False, window=40,
                            max_q=16, max_kv=3000, gen_seed=6)
    yield _fallback_case()


@pytest.mark.parametrize("case", range(4))
def test_static_scratch_entry_matches_the_oracle_and_sdpa_varlen_twice(dev, case):
    call = list(_cases())[case]
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    seq = torch.from_numpy(call.seq_info).to(dev)
    ref, seg_id, st_ref = O.sdpa_varlen(call.q, call.k_store, call.v_store, call.seq_info, call.causal,
                                        call.window, call.scale)
    _, lo, hi, _ = O.visible_interval(call.seq_info, call.T, call.causal, call.window, call.rows, call.cols)
    live = (seg_id >= 0) & (hi > lo)
    empty = (seg_id == O.UNCOVERED) | ((seg_id >= 0) & (hi <= lo))
    gen = pkg.sdpa_varlen(q, k, v, seq, causal=call.causal, window=call.window, scale=call.scale)
    torch.cuda.synchronize()
    for attempt in range(2):
        out = torch.full((call.T, call.Hq, call.D), float("nan"), dtype=torch.bfloat16, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        _static_call(call, q, k, v, seq, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == st_ref, f"call {attempt}: status {int(st.item())} != {st_ref}"
        g = out.double().cpu().numpy()
        if live.any():
            assert np.isfinite(g[live]).all(), f"call {attempt}: non-finite output"
            err = np.abs(g[live] - ref[live])
            assert err.max() <= MAX_ABS, f"call {attempt}: max abs err {err.max():.4g} against the oracle"
            assert err.mean() <= MEAN_ABS, f"call {attempt}: mean abs err {err.mean():.4g} against the oracle"
            d = np.abs(g[live] - gen.double().cpu().numpy()[live])
            assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, f"call {attempt}: differs from sdpa_varlen"
        if empty.any():
            bits = out[torch.as_tensor(np.nonzero(empty)[0], device=dev)].view(torch.int16)
            assert bool((bits == 0).all()), f"call {attempt}: uncovered or keyless rows are not exactly 0"


def test_static_scratch_rejects_sizes_beyond_its_maximum(dev):
    lib, f = _fn()
    dummy = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    seq = torch.zeros((1, 4), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    T = 1 << 22  # far beyond what 32 MiB of scratch can plan for
    p = dummy.data_ptr()
    code = f(p, T, 32, 128, 32 * 128, 128, p, p, 1 << 20, 1, 8, seq.data_ptr(), 1, 1, 0, 0.1, p,
             32 * 128, 128, st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 7  # SDPA_ERR_WORKSPACE, returned before any launch
    msg = lib.sdpa_last_error().decode()
    assert "static scratch holds" in msg and str(32 << 20) in msg
