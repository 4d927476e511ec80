"""Pins for the oracle's dense entry, ``sdpa_causal_prefill``, and for its work counts.

The dense entry is bottom-right causal GQA attention at batch 1: the Lq queries are the last
Lq of Lkv positions ("[CUDA] Use Triton TMA for long-context causal prefill", Operator-level
performance table: B=1 global causal prefill, Hq=16, Hkv=2, Lq < Lkv).  Query i sits at
position Lkv - Lq + i and sees keys 0 .. Lkv - Lq + i.  These checks hold it against things
other than the oracle:

* torch's CPU fp64 ``scaled_dot_product_attention`` with a boolean mask built here from that
  predicate and the KV heads repeated for GQA (``repeat_interleave``), at Lq != Lkv, so that a
  top-left alignment, a dropped causal mask or a transposed head map all fail;
* a scalar triple loop with ``math.exp``;
* mutants of the dense entry (each a plausible slip) that the check must reject;
* the closed form of the useful work: a bottom-right causal row i sees Lkv - Lq + i + 1
  keys, so the rows see Lq*Lkv - Lq*(Lq-1)/2 keys together (8,256 for the 128x128 tiny case,
  8,257,792 for 512x16,384 and 528,484,352 for 4,096x131,072), and the decode batch reads
  kv_end keys per sequence.
"""

import math

import numpy as np
import pytest
import torch

from oracle import sdpa_varlen_oracle as O
from workloads import synth


def _inputs(Lq, Lkv, Hq, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((Lq, Hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((Lkv, Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((Lkv, Hkv, D), generator=g).to(torch.bfloat16)
    return q, k, v


def _torch_bottom_right(q, k, v, scale):
    """torch SDPA in fp64 on the CPU, mask from the predicate j <= Lkv - Lq + i."""
    Lq, Hq, D = q.shape
    Lkv, Hkv, _ = k.shape
    group = Hq // Hkv
    qd = q.double().permute(1, 0, 2)                                 # [Hq, Lq, D]
    kd = k.double().permute(1, 0, 2).repeat_interleave(group, 0)    # [Hq, Lkv, D]
    vd = v.double().permute(1, 0, 2).repeat_interleave(group, 0)
    i = torch.arange(Lq)[:, None]
    j = torch.arange(Lkv)[None, :]
    mask = j <= (Lkv - Lq) + i                                      # [Lq, Lkv]
    o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    o = o.permute(1, 0, 2).numpy()
    # a row that sees nothing (only when Lkv < Lq) is 0 by the oracle's reading; torch
    # returns NaN there, so those rows are compared separately
    empty = (Lkv - Lq + np.arange(Lq)) < 0
    return o, empty


def _scalar(q, k, v, scale):
    Lq, Hq, D = q.shape
    Lkv, Hkv, _ = k.shape
    group = Hq // Hkv
    qf, kf, vf = q.double().tolist(), k.double().tolist(), v.double().tolist()
    out = np.zeros((Lq, Hq, D))
    for i in range(Lq):
        p = Lkv - Lq + i
        for h in range(Hq):
            hk = h // group
            keys = [jj for jj in range(Lkv) if jj <= p]
            if not keys:
                continue
            s = [scale * sum(qf[i][h][d] * kf[jj][hk][d] for d in range(D)) for jj in keys]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for d in range(D):
                out[i, h, d] = sum(e[n] * vf[keys[n]][hk][d] for n in range(len(keys))) / z
    return out


SHAPES = [
    # (Lq, Lkv, Hq, Hkv, D)
    (5, 13, 6, 2, 8),
    (7, 7, 4, 4, 16),
    (1, 9, 8, 2, 8),
    (9, 20, 6, 3, 8),
    (12, 5, 4, 2, 8),  # Lkv < Lq: the first rows see nothing and are 0
]


@pytest.mark.parametrize("shape", SHAPES)
def test_dense_entry_matches_masked_torch_attention(shape):
    Lq, Lkv, Hq, Hkv, D = shape
    q, k, v = _inputs(Lq, Lkv, Hq, Hkv, D, seed=sum(shape))
    scale = 1.0 / math.sqrt(D)
    got = O.sdpa_causal_prefill(q, k, v, scale)
    ref, empty = _torch_bottom_right(q, k, v, scale)
    assert got.shape == (Lq, Hq, D)
    np.testing.assert_allclose(got[~empty], ref[~empty], rtol=0, atol=1e-12)
    assert (got[empty] == 0).all()


@pytest.mark.parametrize("shape", SHAPES[:3])
def test_dense_entry_matches_scalar_loops(shape):
    Lq, Lkv, Hq, Hkv, D = shape
    q, k, v = _inputs(Lq, Lkv, Hq, Hkv, D, seed=7 + sum(shape))
    got = O.sdpa_causal_prefill(q, k, v, 0.3)
    np.testing.assert_allclose(got, _scalar(q, k, v, 0.3), rtol=0, atol=1e-12)


def test_dense_entry_subset_of_rows_leaves_the_rest_zero():
    q, k, v = _inputs(6, 15, 4, 2, 8, seed=3)
    full = O.sdpa_causal_prefill(q, k, v, 0.5)
    part = O.sdpa_causal_prefill(q, k, v, 0.5, rows_subset=[1, 4])
    np.testing.assert_array_equal(part[[1, 4]], full[[1, 4]])
    assert (part[[0, 2, 3, 5]] == 0).all()


# mutants of the dense entry: each a slip the check above must reject
def _mut_top_left(q, k, v, scale):  # segment (0, Lq, 0, Lq): queries at the first positions
    Lq = q.shape[0]
    out, _, _ = O.sdpa_varlen(q, k[:, None], v[:, None], np.array([[0, Lq, 0, Lq]]), True, 0, scale)
    return out


def _mut_not_causal(q, k, v, scale):
    Lq, Lkv = q.shape[0], k.shape[0]
    out, _, _ = O.sdpa_varlen(q, k[:, None], v[:, None], np.array([[0, Lq, 0, Lkv]]), False, 0, scale)
    return out


def _mut_head_axis(q, k, v, scale):  # the store built as [Lkv, Hkv, 1, D]: one KV head per column
    Lq, Lkv = q.shape[0], k.shape[0]
    Hkv = k.shape[1]
    kk, vv = k[:, :, None].expand(-1, -1, Hkv, -1), v[:, :, None].expand(-1, -1, Hkv, -1)
    out, _, _ = O.sdpa_varlen(q, kk.contiguous(), vv.contiguous(), np.array([[0, Lq, 0, Lkv]]), True, 0, scale)
    return out


@pytest.mark.parametrize("mutant", [_mut_top_left, _mut_not_causal, _mut_head_axis])
def test_the_dense_check_rejects_plausible_slips(mutant):
    Lq, Lkv, Hq, Hkv, D = 5, 13, 6, 2, 8
    q, k, v = _inputs(Lq, Lkv, Hq, Hkv, D, seed=11)
    ref, empty = _torch_bottom_right(q, k, v, 0.35)
    assert np.abs(O.sdpa_causal_prefill(q, k, v, 0.35) - ref).max() < 1e-12
    assert np.abs(mutant(q, k, v, 0.35) - ref).max() > 1e-3


# ------------------------------------------------------------------------------------------
# closed forms of the useful work
# ------------------------------------------------------------------------------------------

def _bottom_right_pairs(Lq, Lkv):
    return Lq * Lkv - Lq * (Lq - 1) // 2


@pytest.mark.parametrize("index, Lq, Lkv, pairs", [
    (0, 128, 128, 8_256),
    (1, 512, 16_384, 8_257_792),
    (2, 4_096, 131_072, 528_484_352),
])
def test_useful_flops_of_the_prefill_workloads_in_closed_form(index, Lq, Lkv, pairs):
    assert _bottom_right_pairs(Lq, Lkv) == pairs
    c = synth.workload(index).calls[0]
    assert (c.T, c.rows) == (Lq, Lkv)
    assert O.useful_flops(c.seq_info, c.T, c.Hq, c.D, c.causal, c.window, c.rows, c.cols) == \
        4 * c.D * c.Hq * pairs


def test_useful_flops_of_the_d64_prefill_is_33_82_gflop():
    c = synth.workload(1).calls[0]
    f = O.useful_flops(c.seq_info, c.T, c.Hq, c.D, c.causal, c.window, c.rows, c.cols)
    assert f == 33_823_916_032  # 4 * 64 * 16 * 8,257,792


def test_useful_kv_bytes_of_the_decode_batch_in_closed_form():
    c = synth.workload(3).calls[0]
    kv_end = c.seq_info[:, 3].astype(np.int64)
    # K and V, Hkv heads of D bf16 values per visible position: 1 KiB per position here
    assert c.Hkv * c.D * 2 * 2 == 1024
    assert O.useful_kv_bytes(c.seq_info, c.T, c.Hkv, c.D, c.window, c.rows, c.cols) == int(kv_end.sum()) * 1024
    # one query per sequence, causal at the last position: it sees all kv_end keys
    assert O.useful_flops(c.seq_info, c.T, c.Hq, c.D, True, 0, c.rows, c.cols) == \
        4 * c.D * c.Hq * int(kv_end.sum())
