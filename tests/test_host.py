"""Host-side checks that need no GPU: the library builds/loads, exports every symbol the
header declares, and rejects bad arguments before making any CUDA call.

Only argument errors that the C interface detects ahead of any CUDA call are exercised
here (the pointers are fake but never dereferenced); nothing launches a kernel.
"""

import os
import re

import pytest

import varlen_gqa_attention_gb300 as pkg
from varlen_gqa_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa_varlen.h")

FAKE = 0x10000  # 16-byte aligned, never dereferenced


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdpa_[a-z_]+)\s*\(", text)))


def test_library_builds_in_tree_and_loads():
    path = _build.build()
    assert os.path.exists(path)
    assert os.path.commonpath([path, ROOT]) == ROOT
    lib = pkg.library()
    assert lib.sdpa_version() == 100


def test_every_declared_symbol_is_exported():
    lib = pkg.library()
    names = _declared_functions()
    assert set(names) >= {"sdpa_varlen", "sdpa_causal_prefill", "sdpa_varlen_workspace_bytes",
                          "sdpa_last_error", "sdpa_set_route_policy", "sdpa_version"}
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(pkg.EXPORTS) == sorted(names)


def test_status_bits_match_the_oracle_constants():
    from oracle import sdpa_varlen_oracle as O

    assert (pkg.SEG_BAD_QRANGE, pkg.SEG_BAD_COL, pkg.SEG_BAD_KV, pkg.SEG_SPAN, pkg.SEG_OVERLAP) == \
        (O.SEG_BAD_QRANGE, O.SEG_BAD_COL, O.SEG_BAD_KV, O.SEG_SPAN, O.SEG_OVERLAP)
    text = open(HEADER).read()
    for name, val in (("SDPA_SEG_BAD_QRANGE", 1), ("SDPA_SEG_BAD_COL", 2), ("SDPA_SEG_BAD_KV", 4),
                      ("SDPA_SEG_SPAN", 8), ("SDPA_SEG_OVERLAP", 16), ("SDPA_DEV_TIMEOUT", 32)):
        assert re.search(rf"#define {name} {val}\b", text), name


def _call(**kw):
    a = dict(q=FAKE, T=8, Hq=4, D=64, q_rs=256, q_hs=64, k=FAKE, v=FAKE, rows=16, cols=2, Hkv=2,
             seq=FAKE, S=1, causal=1, window=0, scale=0.125, out=FAKE, o_rs=256, o_hs=64, ws=FAKE,
             ws_bytes=1 << 30, status=None, stream=None)
    a.update(kw)
    lib = pkg.library()
    code = lib.sdpa_varlen(a["q"], a["T"], a["Hq"], a["D"], a["q_rs"], a["q_hs"], a["k"], a["v"],
                           a["rows"], a["cols"], a["Hkv"], a["seq"], a["S"], a["causal"], a["window"],
                           a["scale"], a["out"], a["o_rs"], a["o_hs"], a["ws"], a["ws_bytes"],
                           a["status"], a["stream"])
    return code, lib.sdpa_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), 3), (dict(D=0), 3), (dict(Hq=6, Hkv=4), 4), (dict(Hq=256, Hkv=1), 4),
    (dict(T=-1), 2), (dict(S=-1), 2), (dict(rows=0), 2), (dict(cols=0), 2), (dict(Hkv=0), 2),
    (dict(window=-3), 8), (dict(scale=float("inf")), 8), (dict(scale=float("nan")), 8),
    (dict(q=None), 1), (dict(out=None), 1), (dict(seq=None), 1), (dict(ws=None), 7),
    (dict(q=FAKE + 2), 6), (dict(out=FAKE + 8), 6), (dict(q_rs=250), 5), (dict(o_hs=3), 5),
    (dict(ws=FAKE + 16), 6),
])
def test_bad_arguments_are_rejected_before_any_cuda_call(kw, code):
    got, msg = _call(**kw)
    assert got == code, msg
    assert msg


def test_route_policy_is_checked():
    lib = pkg.library()
    assert lib.sdpa_set_route_policy(7) == 8
    assert lib.sdpa_set_route_policy(0) == 0


def test_workspace_query_depends_only_on_sizes():
    a = pkg.workspace_bytes(4096, 16, 2, 128, 1)
    b = pkg.workspace_bytes(4096, 16, 2, 128, 1)
    assert a == b and a > 0 and a % 256 == 0
    assert pkg.workspace_bytes(8192, 16, 2, 128, 1) > a
    assert pkg.workspace_bytes(16, 16, 3, 128, 1) == 0  # Hq % Hkv != 0
    assert pkg.workspace_bytes(16, 16, 2, 80, 1) == 0


def test_product_path_does_not_import_the_oracle():
    src_dir = os.path.join(ROOT, "varlen_gqa_attention_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower().replace("oracles", ""), f


def test_seq_clone_rejects_bad_arguments_before_touching_the_device():
    import varlen_gqa_attention_gb300 as pkg
    lib = pkg.library()
    NULL, SHAPE, HEAD_DIM, ALIGN, ARG = 1, 2, 3, 6, 8  # sdpa_status codes of the header
    p = 1 << 20  # a 16-byte aligned address that is never dereferenced
    assert lib.sdpa_seq_clone(None, p, 8, 2, 1, 128, 0, 1, 4, None) == NULL
    assert lib.sdpa_seq_clone(p + 2, p, 8, 2, 1, 128, 0, 1, 4, None) == ALIGN
    assert lib.sdpa_seq_clone(p, p, 0, 2, 1, 128, 0, 1, 4, None) == SHAPE
    assert lib.sdpa_seq_clone(p, p, 8, 2, 1, 128, 0, 1, -1, None) == SHAPE
    assert lib.sdpa_seq_clone(p, p, 8, 2, 1, 96, 0, 1, 4, None) == HEAD_DIM
    assert lib.sdpa_seq_clone(p, p, 8, 2, 1, 128, 0, 2, 4, None) == ARG
    assert lib.sdpa_seq_clone(p, p, 8, 2, 1, 128, 1, 1, 4, None) == pkg.SDPA_OK  # same column
    assert lib.sdpa_seq_clone(p, p, 8, 2, 1, 128, 0, 1, 0, None) == pkg.SDPA_OK  # empty prefix


def test_prefill_availability_rejects_unknown_head_dims_before_any_cuda_call():
    lib = pkg.library()
    assert lib.sdpa_prefill_available(96) == -1
    assert "head dim 96" in lib.sdpa_last_error().decode()


def _call_modes(seg_mode, S=1):
    lib = pkg.library()
    code = lib.sdpa_varlen_modes(FAKE, 8, 4, 64, 256, 64, FAKE, FAKE, 16, 2, 2, FAKE, seg_mode, S, 0.125,
                                 FAKE, 256, 64, FAKE, 1 << 30, None, None)
    return code, lib.sdpa_last_error().decode()


def test_per_segment_mode_table_is_checked_before_any_cuda_call():
    assert _call_modes(None)[0] == 1          # SDPA_ERR_NULL
    code, msg = _call_modes(FAKE + 8)         # not 16-byte aligned
    assert code == 6 and "seg_mode" in msg    # SDPA_ERR_ALIGN


def _call_static(**kw):
    a = dict(q=FAKE, T=8, Hq=4, D=64, q_rs=256, q_hs=64, k=FAKE, v=FAKE, rows=16, cols=2, Hkv=2,
             seq=FAKE, S=1, causal=1, window=0, scale=0.125, out=FAKE, o_rs=256, o_hs=64, status=None,
             stream=None)
    a.update(kw)
    lib = pkg.library()
    code = lib.sdpa_varlen_splitk_static(a["q"], a["T"], a["Hq"], a["D"], a["q_rs"], a["q_hs"], a["k"], a["v"],
                                         a["rows"], a["cols"], a["Hkv"], a["seq"], a["S"], a["causal"],
                                         a["window"], a["scale"], a["out"], a["o_rs"], a["o_hs"], a["status"],
                                         a["stream"])
    return code, lib.sdpa_last_error().decode()


@pytest.mark.parametrize("kw", [
    dict(D=96), dict(Hq=6, Hkv=4), dict(Hq=256, Hkv=1), dict(T=-1), dict(S=-1), dict(rows=0), dict(cols=0),
    dict(window=-3), dict(scale=float("nan")), dict(q=None), dict(out=None), dict(seq=None),
    dict(q=FAKE + 2), dict(out=FAKE + 8), dict(q_rs=250), dict(o_hs=3),
    dict(T=(1 << 40) // 64 + 1, Hq=128, Hkv=1),  # Hq * T beyond 2^40
])
def test_static_entry_rejects_what_sdpa_varlen_rejects_with_the_same_message(kw):
    code, msg = _call_static(**kw)
    ref_code, ref_msg = _call(**kw)
    assert code == ref_code and code != 0, (code, msg)
    assert msg == ref_msg


def test_workspace_status_checks_its_arguments_before_any_cuda_call():
    import ctypes

    lib = pkg.library()
    v = ctypes.c_int32(0)
    assert lib.sdpa_workspace_status(None, 1 << 20, ctypes.byref(v), None) == 1
    assert lib.sdpa_workspace_status(FAKE, 1 << 20, None, None) == 1
    assert lib.sdpa_workspace_status(FAKE + 16, 1 << 20, ctypes.byref(v), None) == 6
    assert lib.sdpa_workspace_status(FAKE, 8, ctypes.byref(v), None) == 7


def _cpu_args(**kw):
    import torch

    a = dict(q=torch.zeros(8, 4, 64, dtype=torch.bfloat16), k=torch.zeros(16, 2, 2, 64, dtype=torch.bfloat16),
             v=torch.zeros(16, 2, 2, 64, dtype=torch.bfloat16), seq=torch.zeros(1, 4, dtype=torch.int32))
    a.update(kw)
    return a


def _bad_inputs():
    import torch

    bf = torch.bfloat16
    return [
        ("fp16 q", _cpu_args(q=torch.zeros(8, 4, 64, dtype=torch.float16)), "q must be bf16"),
        ("fp32 store", _cpu_args(k=torch.zeros(16, 2, 2, 64)), "k_store must be bf16"),
        ("int64 table", _cpu_args(seq=torch.zeros(1, 4, dtype=torch.int64)), "seq_info"),
        ("table of 3 columns", _cpu_args(seq=torch.zeros(1, 3, dtype=torch.int32)), "seq_info"),
        ("strided store", _cpu_args(k=torch.zeros(16, 4, 2, 64, dtype=bf)[:, ::2],
                                    v=torch.zeros(16, 4, 2, 64, dtype=bf)[:, ::2]), "contiguous"),
        ("q inner stride 2", _cpu_args(q=torch.zeros(8, 4, 128, dtype=bf)[:, :, ::2]), "inner stride"),
        ("head dims differ", _cpu_args(q=torch.zeros(8, 4, 128, dtype=bf)), "head dims"),
        ("3-d store", _cpu_args(k=torch.zeros(16, 2, 64, dtype=bf), v=torch.zeros(16, 2, 64, dtype=bf)), "stores"),
        ("host tensors", _cpu_args(), "CUDA device"),
    ]


@pytest.mark.parametrize("entry", ["sdpa_varlen", "sdpa_varlen_splitk_static", "sdpa_varlen_modes",
                                   "sdpa_varlen_append"])
def test_python_entries_reject_bad_tensors_before_the_library_call(entry):
    import torch

    for what, a, needle in _bad_inputs():
        f = getattr(pkg, entry)
        with pytest.raises(ValueError) as ei:
            if entry == "sdpa_varlen_modes":
                f(a["q"], a["k"], a["v"], a["seq"], torch.zeros(a["seq"].shape[0], 2, dtype=torch.int32))
            elif entry == "sdpa_varlen_append":
                kn = torch.zeros(a["q"].shape[0], a["k"].shape[-2] if a["k"].dim() == 4 else 2, a["q"].shape[-1],
                                 dtype=torch.bfloat16)
                f(a["q"], kn, kn, a["k"], a["v"], a["seq"], causal=True)
            else:
                f(a["q"], a["k"], a["v"], a["seq"], causal=True)
        assert needle in str(ei.value), (entry, what, str(ei.value))


def test_python_static_entry_checks_out_and_status():
    import torch

    a = _cpu_args()
    with pytest.raises(ValueError, match="out must be bf16"):
        pkg.sdpa_varlen_splitk_static(a["q"], a["k"], a["v"], a["seq"], causal=True,
                                      out=torch.zeros(8, 4, 32, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="seg_mode"):
        pkg.sdpa_varlen_modes(a["q"], a["k"], a["v"], a["seq"], torch.zeros(1, 3, dtype=torch.int32))
