"""The causal tile skip, counted on the device.

fa_fwd_counted / fa_bwd_counted report, per sequence, how many (query tile,
key tile) pairs the kernels actually computed scores for, counted by the
thread that issues the score products.  Under the causal mask the tiles wholly
above the diagonal must be skipped ("Attention 算子优化…", section 四), so the
counts must equal the oracle's brute-force enumeration of tiles holding at
least one visible score, times the number of query heads, bit for bit.  The
outputs of the counted calls are also checked against the plain entry points'.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs, make_qkv
from tests.gpu_util import fa_module

pytestmark = pytest.mark.gpu


def _device_inputs(t, lengths, dev):
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    return q, k, v, cu


def _fwd_counts(fa, q, k, v, cu, lengths, causal, scale):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    B, N = len(lengths), max(max(lengths), 1)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    counts = torch.full((B,), -1, dtype=torch.int64, device=q.device)
    fa.fa_fwd_counted(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu, counts)
    fa.fa_stream_status()
    o_plain, lse_plain = fa.attention_forward(q, k, v, causal, scale=scale, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    assert torch.equal(o.view(torch.int16), o_plain.view(torch.int16))
    assert torch.equal(lse, lse_plain)
    return counts.cpu().tolist(), o, lse


@pytest.mark.parametrize("name", ["fwd_b2_h32_n4096_d128_causal", "fwd_varlen8_hq32_hkv8_d128_causal",
                                  "fwd_b4_h16_n2048_d64", "fwdbwd_b2_h16_n4096_d64_causal"])
def test_forward_tile_counts_match_oracle(cuda_device, name):
    fa = fa_module()
    w = WORKLOADS[name]
    t = make_inputs(w, with_do=False)
    lengths = w.seq_lengths
    q, k, v, cu = _device_inputs(t, lengths, cuda_device)
    got, _, _ = _fwd_counts(fa, q, k, v, cu, lengths, w.causal, w.scale)
    want = [w.Hq * n for n in oracle.tile_counts(lengths, w.causal)]
    assert got == want, (got, want)
    if w.causal:
        # about half of the full grid: the tiles on and below the diagonal
        full = [w.Hq * (-(-L // 128)) ** 2 for L in lengths]
        assert all(2 * g > f for g, f in zip(got, full))
        assert all(g < f for g, f in zip(got, full))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_tile_counts_ragged_packs(cuda_device, d, causal):
    """Short, empty and one-token sequences, GQA: a sequence with no tokens
    counts nothing, one with a partial tile counts that tile."""
    fa = fa_module()
    lengths = [5, 1, 300, 128, 129, 0, 640, 77]
    t = make_qkv(sum(lengths), 4, 1, d, seed=40, with_do=True)
    q, k, v, cu = _device_inputs(t, lengths, cuda_device)
    got, o, lse = _fwd_counts(fa, q, k, v, cu, lengths, causal, d ** -0.5)
    want = [4 * n for n in oracle.tile_counts(lengths, causal)]
    assert got == want, (got, want)
    # the backward's gradient kernel walks the same pairs, key tile outermost
    do = t["do"].to(cuda_device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    T, Hq, _ = q.shape
    ws = torch.empty(fa.fa_bwd_workspace_size(Hq, T, d), dtype=torch.uint8, device=cuda_device)
    counts = torch.full((len(lengths),), -1, dtype=torch.int64, device=cuda_device)
    fa.fa_bwd_counted(q, k, v, o, do, lse, dq, dk, dv, len(lengths), Hq, 1, max(lengths), d, T, d ** -0.5, causal,
                      cu, ws, counts)
    fa.fa_stream_status()
    assert counts.cpu().tolist() == want


@pytest.mark.parametrize("name", ["fwdbwd_b2_h16_n4096_d64_causal", "fwdbwd_b2_h32_n4096_d128_causal"])
def test_backward_tile_counts_match_oracle(cuda_device, name):
    fa = fa_module()
    w = WORKLOADS[name]
    t = make_inputs(w)
    lengths = w.seq_lengths
    q, k, v, cu = _device_inputs(t, lengths, cuda_device)
    do = t["do"].to(cuda_device)
    T, Hq, d = q.shape
    o, lse = fa.attention_forward(q, k, v, w.causal, cu_seqlens=cu, max_seqlen=w.N)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(Hq, T, d), dtype=torch.uint8, device=cuda_device)
    counts = torch.full((len(lengths),), -1, dtype=torch.int64, device=cuda_device)
    fa.fa_bwd_counted(q, k, v, o, do, lse, dq, dk, dv, len(lengths), Hq, w.Hkv, w.N, d, T, w.scale, w.causal, cu,
                      ws, counts)
    fa.fa_stream_status()
    want = [w.Hq * n for n in oracle.tile_counts(lengths, w.causal)]
    assert counts.cpu().tolist() == want
    # dK and dV come out of the counted call bit for bit as from the plain one
    ref = fa.attention_backward(q, k, v, o, lse, do, w.causal, cu_seqlens=cu, max_seqlen=w.N)
    fa.fa_stream_status()
    assert torch.equal(dk.view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(dv.view(torch.int16), ref[2].view(torch.int16))
