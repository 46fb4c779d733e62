"""GPU parity of the forward kernel against the fp64 oracle.

Small and odd shapes (several tiles plus a ragged tail) are compared element
by element; the full-size workloads are compared on sampled rows, which the
oracle evaluates one by one, plus properties that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs, make_qkv
from tests.golden_io import load
from tests.gpu_util import assert_fwd_close, cu_of, f64, run_fwd

pytestmark = pytest.mark.gpu


def check_case(T, Hq, Hkv, d, causal, lengths=None, N=None, seed=0, q_mult=1.0):
    t = make_qkv(T, Hq, Hkv, d, seed=seed, q_mult=q_mult)
    o, lse = run_fwd(t["q"], t["k"], t["v"], causal, lengths=lengths, N=N)
    cu = cu_of(T, lengths, N)
    o_ref, lse_ref = oracle.attention_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), cu, d ** -0.5, causal)
    return assert_fwd_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 127, 128, 129, 300, 512])
def test_fwd_single_sequence(cuda_device, d, causal, N):
    check_case(N, 2, 2, d, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_batched_gqa(cuda_device, d, causal):
    check_case(3 * 384, 8, 2, d, causal, N=384, seed=1)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_packed_ragged(cuda_device, d, causal):
    lengths = [5, 1, 300, 128, 129, 0, 640, 77]
    check_case(sum(lengths), 4, 1, d, causal, lengths=lengths, seed=2)


def test_fwd_wide_scores_stay_finite(cuda_device):
    """Queries scaled by 8: the softmax is nearly one-hot, so O is close to a
    single V row and |O| reaches 4-5.  Rounding O to bf16 (8 significant
    bits) then costs up to 2^-9 |O| on its own, above the 1e-2 absolute bound
    the N(0,1) workloads use, so this case allows 1e-2 + 2^-8 |O_ref| per
    element (one more half-ulp of headroom for the accumulation)."""
    t = make_qkv(600, 2, 2, 64, seed=3, q_mult=8.0)
    o, lse = run_fwd(t["q"], t["k"], t["v"], True)
    o_ref, lse_ref = oracle.attention_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), [0, 600], 0.125, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert (np.abs(o - o_ref) <= 1e-2 + 2.0 ** -8 * np.abs(o_ref)).all()
    assert np.abs(o - o_ref).mean() <= 1e-3
    assert np.abs(lse - lse_ref).max() <= 1e-3


def test_fwd_workload_small(cuda_device):
    """B=1, H=1, N=256, d=64, non-causal, seed 0: every output element."""
    w = WORKLOADS["fwd_b1_h1_n256_d64"]
    t = make_inputs(w)
    o, lse = run_fwd(t["q"], t["k"], t["v"], w.causal, N=w.N)
    o_ref, lse_ref = oracle.attention_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), cu_of(w.T, N=w.N),
                                              w.scale, w.causal)
    assert_fwd_close(o, lse, o_ref, lse_ref)


def _pad_to(x, d):
    out = np.zeros((x.shape[0], 1, d))
    out[:, 0, : x.shape[1]] = x
    return torch.tensor(out, dtype=torch.bfloat16)


def test_fwd_online_softmax_worked_examples(cuda_device):
    """The pages' worked examples, zero-padded to d = 64 (exact in bf16)."""
    g = load("online_softmax_two_blocks.txt")
    scores = g["scores_block1"] + g["scores_block2"]
    n = len(scores)
    q = _pad_to(np.ones((n, 1)), 64)
    k = _pad_to(np.array(scores, float)[:, None], 64)
    v = _pad_to(np.zeros((n, 1)), 64)
    _, lse = run_fwd(q, k, v, False, scale=1.0)
    # LSE = m + ln l with m = 3 and the page's sum l about m = 3
    assert abs(lse[0, 0] - (3 + math.log(g["exact_l_new"]))) <= 1e-3
    g = load("online_softmax_value_example.txt")
    n = len(g["scores"])
    q = _pad_to(np.ones((n, 1)), 64)
    k = _pad_to(np.array(g["scores"], float)[:, None], 64)
    v = _pad_to(np.array(g["values"], float)[:, None], 64)
    o, lse = run_fwd(q, k, v, False, scale=1.0)
    want = g["merged_u"] / g["merged_l"]
    assert abs(o[0, 0, 0] - want) <= 0.125 + 1e-3 * want  # bf16 output spacing at 25.75 is 0.125
    assert abs(lse[0, 0] - (3 + math.log(g["merged_l"]))) < 1e-3


def test_fwd_hand_causal_prefix_means(cuda_device):
    """Q = 0, causal: O_i = mean(V[0..i]), LSE_i = ln(i + 1)."""
    L = 200
    q = torch.zeros(L, 1, 64, dtype=torch.bfloat16)
    k = make_qkv(L, 1, 1, 64, seed=4)["k"]
    vv = np.zeros((L, 1, 64))
    vv[:, 0, 0] = np.arange(L) % 7
    vv[:, 0, 1] = 1.0
    v = torch.tensor(vv, dtype=torch.bfloat16)
    o, lse = run_fwd(q, k, v, True)
    want = np.cumsum(vv[:, 0, 0]) / np.arange(1, L + 1)
    np.testing.assert_allclose(o[:, 0, 0], want, atol=1e-2)
    np.testing.assert_allclose(o[:, 0, 1], 1.0, atol=4e-3)
    np.testing.assert_allclose(lse[0], np.log(np.arange(1, L + 1)), atol=1e-3)


def _whole_heads_check(t, o, lse, w, cu, pairs):
    """Every row of the given (sequence, query head) pairs against the oracle
    on that slice alone, at the forward bars."""
    group = w.Hq // w.Hkv
    for s, h in pairs:
        a, b = int(cu[s]), int(cu[s + 1])
        kvh = h // group
        o_ref, lse_ref = oracle.attention_forward(f64(t["q"][a:b, h:h + 1]), f64(t["k"][a:b, kvh:kvh + 1]),
                                                  f64(t["v"][a:b, kvh:kvh + 1]), [0, b - a], w.scale, w.causal)
        assert_fwd_close(o[a:b, h:h + 1], lse[h:h + 1, a:b], o_ref, lse_ref)


def _sampled_rows_check(w, whole_pairs, n_rows=384, seed=123):
    t = make_inputs(w)
    o, lse = run_fwd(t["q"], t["k"], t["v"], w.causal,
                     lengths=w.seq_lengths if w.varlen else None, N=None if w.varlen else w.N)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vmax = float(t["v"].float().abs().max())
    assert np.abs(o).max() <= vmax * (1 + 2 ** -7)
    r = np.random.default_rng(seed)
    cu = cu_of(w.T, w.seq_lengths if w.varlen else None, None if w.varlen else w.N)
    _whole_heads_check(t, o, lse, w, cu, whole_pairs)
    # include every sequence's first and last rows and the tile edges
    toks = list(r.integers(0, w.T, n_rows))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        toks += [a, b - 1, min(a + 127, b - 1), min(a + 128, b - 1)]
    toks = np.array(toks)
    heads = r.integers(0, w.Hq, len(toks))
    qf, kf, vf = f64(t["q"]), f64(t["k"]), f64(t["v"])
    o_ref, lse_ref = oracle.attention_forward_rows(qf, kf, vf, cu, w.scale, w.causal, toks, heads)
    err = np.abs(o[toks, heads] - o_ref)
    assert err.max() <= 1e-2, err.max()
    assert err.mean() <= 1e-3, err.mean()
    assert np.abs(lse[heads, toks] - lse_ref).max() <= 1e-3


def test_fwd_workload_b4_h16_n2048_d64(cuda_device):
    """Full element-by-element comparison (the oracle finishes in seconds)."""
    w = WORKLOADS["fwd_b4_h16_n2048_d64"]
    t = make_inputs(w)
    o, lse = run_fwd(t["q"], t["k"], t["v"], w.causal, N=w.N)
    o_ref, lse_ref = oracle.attention_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), cu_of(w.T, N=w.N),
                                              w.scale, w.causal)
    assert_fwd_close(o, lse, o_ref, lse_ref)


def test_fwd_workload_b2_h32_n4096_d128_causal(cuda_device):
    """Sampled rows over the whole output, plus two whole (sequence, head)
    slices, every row."""
    _sampled_rows_check(WORKLOADS["fwd_b2_h32_n4096_d128_causal"], whole_pairs=[(0, 0), (1, 31)])


def test_fwd_workload_varlen_gqa(cuda_device):
    """Sampled rows, plus whole slices: the longest sequence (6860 tokens) on
    the last head of the last K/V group, and a short one (1178) on head 5."""
    _sampled_rows_check(WORKLOADS["fwd_varlen8_hq32_hkv8_d128_causal"], whole_pairs=[(7, 31), (6, 5)])


def test_fwd_bad_packed_offsets_are_reported(cuda_device):
    """Offsets past T are caught on the device and reported, nothing written."""
    import exact_attention_21_gb300.fa as fa
    t = make_qkv(256, 1, 1, 64, seed=5)
    dev = torch.device("cuda:0")
    q, k, v = (x.to(dev) for x in (t["q"], t["k"], t["v"]))
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 256, device=dev)
    cu = torch.tensor([0, 100, 400], dtype=torch.int32, device=dev)
    fa.fa_fwd(q, k, v, o, lse, 2, 1, 1, 300, 64, 256, 0.125, 1, cu)
    with pytest.raises(fa.FAError) as ei:
        fa.fa_stream_status()
    assert ei.value.code == fa.FA_ERR_INVALID_ARG
    fa.fa_stream_status()  # cleared
