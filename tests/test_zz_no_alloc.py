"""The allocation-free entry point, sdpa_varlen_splitk_static.

Some callers cannot allocate device memory (a runtime with a fixed memory plan, a plugin
that must not call cudaMalloc, a binding with no device allocator), so they cannot hand
sdpa_varlen a workspace.  sdpa_varlen_splitk_static keeps its scratch in a static device
array of the library instead.  These tests call it through the C interface (ctypes, no
torch allocation on its path) and check it against sdpa_varlen on the same inputs, twice
in a row (the second call finds the first call's leftovers in the shared array).  This file
is collected last so that a failure here cannot hide the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import varlen_gqa_attention_gb300 as pkg
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


def _cases():
    rng = np.random.default_rng(21)
    yield synth.batched_decode(seed=2).calls[0]
    yield synth.random_call(rng, D=128, Hq=16, Hkv=2, T=96, S=6, rows=1500, cols=7, causal=True, window=0,
                            max_q=20, max_kv=1500, gen_seed=5)
    yield synth.random_call(rng, D=64, Hq=8, Hkv=2, T=64, S=5, rows=300, cols=6, causal=False, window=40,
                            max_q=16, max_kv=3000, gen_seed=6)


@pytest.mark.parametrize("case", range(3))
def test_static_scratch_entry_matches_sdpa_varlen_twice(dev, case):
    call = list(_cases())[case]
    q, k, v = call.q.to(dev), call.k_store.to(dev), call.v_store.to(dev)
    seq = torch.from_numpy(call.seq_info).to(dev)
    st_ref = torch.zeros(1, dtype=torch.int32, device=dev)
    ref = pkg.sdpa_varlen(q, k, v, seq, causal=call.causal, window=call.window, scale=call.scale, status=st_ref)
    torch.cuda.synchronize()
    ref64 = ref.double()
    for attempt in range(2):
        out = torch.full_like(ref, float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        _static_call(call, q, k, v, seq, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == int(st_ref.item())
        err = (out.double() - ref64).abs()
        assert torch.isfinite(out.double()).all(), f"call {attempt}: non-finite output"
        assert float(err.max()) <= MAX_ABS, f"call {attempt}: max abs diff {float(err.max()):.4g}"
        assert float(err.mean()) <= MEAN_ABS, f"call {attempt}: mean abs diff {float(err.mean()):.4g}"
        zero_ref = (ref.view(torch.int16) == 0).all(dim=-1)
        zero_out = (out.view(torch.int16) == 0).all(dim=-1)
        assert bool((zero_ref == zero_out).all()), f"call {attempt}: zero rows differ"


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
