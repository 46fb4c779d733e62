"""GPU parity of the split-K/V decoding path against the fp64 oracle.

One new query per sequence against a K/V cache: small and odd cache lengths
(several 128-key tiles plus a ragged tail, empty caches), every supported GQA
group, long caches that the library cuts into many splits, and the full-size
decoding workloads.  The bar is the forward's: max |dO| <= 1e-2,
mean |dO| <= 1e-3, max |dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import WORKLOADS, make_decode_qkv, make_inputs
from tests.gpu_util import assert_fwd_close, f64, fa_module

pytestmark = pytest.mark.gpu


def run_decode(t, lengths=None, N=None):
    fa = fa_module()
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev).contiguous() for n in ("q", "k", "v"))
    if lengths is None:
        cu = None
    else:
        N = max(max(lengths), 1)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o, lse = fa.attention_decode(q, k, v, cu_seqlens_k=cu, max_seqlen_k=N)
    fa.fa_stream_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(B, Hq, Hkv, d, lengths, batched=False, seed=0, q_mult=1.0):
    T = int(sum(lengths))
    t = make_decode_qkv(B, Hq, T, Hkv, d, seed=seed)
    if q_mult != 1.0:
        t["q"] = (t["q"].float() * q_mult).to(torch.bfloat16)
    if batched:
        o, lse = run_decode(t, N=lengths[0])
    else:
        o, lse = run_decode(t, lengths=lengths)
    cu = oracle.cu_from_lengths(lengths)
    o_ref, lse_ref = oracle.attention_decode(f64(t["q"]), f64(t["k"]), f64(t["v"]), cu, d ** -0.5)
    return assert_fwd_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 5, 127, 128, 129, 300, 1000])
def test_decode_batched(cuda_device, d, N):
    check(3, 8, 2, d, [N] * 3, batched=True, seed=N)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [200, 256])
def test_decode_batched_one_split_per_row(cuda_device, d, N):
    """Many short batched caches (64 sequences of two tiles, Hq64/Hkv8): the
    split model gives each (sequence, K/V head) a single split, so the split
    kernel writes O and the LSE itself and no combine runs (d = 64 on head
    pairs, d = 128 unpaired)."""
    check(64, 64, 8, d, [N] * 64, batched=True, seed=N + d)


@pytest.mark.parametrize("heads", [(8, 2), (32, 2)])
def test_decode_many_items_per_cta(cuda_device, heads):
    """Many more (split, K/V head, sequence) items than SMs, of mixed and
    empty lengths: each CTA of the persistent kernel runs a dozen items back
    to back, carrying its rings, its S^T and O^T buffers and the next item's
    query across them (GQA groups of 4 and 16)."""
    lengths = [int(x) for x in np.random.default_rng(31).integers(0, 700, size=160)]
    check(len(lengths), heads[0], heads[1], 128, lengths, seed=31)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_more_sequences_than_the_compact_table(cuda_device, d):
    """1100 packed caches (above the 1024 sequences whose split counts the
    kernel numbers compactly): the split-major numbering, with empty caches."""
    lengths = [int(x) for x in np.random.default_rng(34).integers(0, 300, size=1100)]
    check(len(lengths), 4, 2, d, lengths, seed=34)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_packed_ragged_with_empty_caches(cuda_device, d):
    lengths = [5, 1, 300, 128, 129, 0, 640, 77, 2000]
    o_err = check(len(lengths), 8, 2, d, lengths, seed=5)
    assert o_err is not None


@pytest.mark.parametrize("heads", [(4, 4), (6, 2), (24, 8), (32, 4), (32, 2)])
def test_decode_gqa_groups(cuda_device, heads):
    """Groups 1, 3 (rounded up to 4 inside the kernel), 3, 8 and 16."""
    Hq, Hkv = heads
    check(2, Hq, Hkv, 128, [700, 1500], seed=Hq + Hkv)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_long_cache_many_splits(cuda_device, d):
    """One sequence with a 20k-token cache: the split length the library
    picks gives many splits, which the combine merges."""
    check(1, 4, 1, d, [20000], batched=True, seed=7)


@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (8, 4), (16, 2), (64, 8)])
def test_decode_d64_head_pairs(cuda_device, heads):
    """d = 64 with an even number of K/V heads and groups of 1-8: adjacent K/V
    heads are paired and run on the tensor-core kernel (each query head's
    scores and output come only from its own K/V head), ragged lengths."""
    Hq, Hkv = heads
    check(3, Hq, Hkv, 64, [1, 700, 129], seed=40 + Hq)


@pytest.mark.parametrize("heads", [(3, 3), (32, 2), (9, 1)])
def test_decode_d64_cuda_core_fallback(cuda_device, heads):
    """d = 64 that cannot be paired (odd Hkv, or a group above 8): the
    CUDA-core split kernel."""
    Hq, Hkv = heads
    check(2, Hq, Hkv, 64, [300, 1000], seed=50 + Hq)


def test_decode_d64_many_items_per_cta(cuda_device):
    lengths = [int(x) for x in np.random.default_rng(32).integers(0, 700, size=160)]
    check(len(lengths), 8, 2, 64, lengths, seed=32)


def test_decode_wide_scores_stay_finite(cuda_device):
    """Queries scaled by 8: nearly one-hot weights (see the forward's test for
    the bf16 rounding allowance on |O| of 4-5)."""
    lengths = [900, 3000]
    t = make_decode_qkv(2, 4, sum(lengths), 1, 64, seed=9)
    t["q"] = (t["q"].float() * 8.0).to(torch.bfloat16)
    o, lse = run_decode(t, lengths=lengths)
    o_ref, lse_ref = oracle.attention_decode(f64(t["q"]), f64(t["k"]), f64(t["v"]),
                                             oracle.cu_from_lengths(lengths), 0.125)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert (np.abs(o - o_ref) <= 1e-2 + 2.0 ** -8 * np.abs(o_ref)).all()
    assert np.abs(lse - lse_ref).max() <= 1e-3


def test_decode_matches_last_row_of_the_forward(cuda_device):
    """The decode path and the tiled forward agree on the newest token of
    each sequence (causal forward over the same packed sequences)."""
    fa = fa_module()
    from exact_attention_21_gb300.inputs import make_qkv
    lengths = [130, 1, 700]
    T = sum(lengths)
    t = make_qkv(T, 8, 2, 128, seed=11)
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o_f, l_f = fa.attention_forward(q, k, v, True, cu_seqlens=cu, max_seqlen=max(lengths))
    last = torch.tensor(np.cumsum(lengths) - 1, device=dev)
    o_d, l_d = fa.attention_decode(q[last].contiguous(), k, v, cu_seqlens_k=cu, max_seqlen_k=max(lengths))
    fa.fa_stream_status()
    assert (o_d.float() - o_f[last].float()).abs().max().item() <= 2e-2
    assert (l_d - l_f[:, last]).abs().max().item() <= 2e-3


@pytest.mark.parametrize("name", ["decode_varlen8_hq32_hkv8_d128", "decode_b64_hq64_hkv8_n4096_d128",
                                  "decode_b64_hq64_hkv8_n4096_d64"])
def test_decode_workload(cuda_device, name):
    """Full-size decoding workloads; the 64-sequence one is checked on three
    whole sequences (every head) against the oracle, the packed one in full."""
    w = WORKLOADS[name]
    t = make_inputs(w)
    o, lse = run_decode(t, lengths=w.seq_lengths if w.varlen else None, N=w.N)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    cu = oracle.cu_from_lengths(w.seq_lengths)
    seqs = range(w.B) if w.varlen else [0, 17, w.B - 1]
    for b in seqs:
        a, e = int(cu[b]), int(cu[b + 1])
        o_ref, lse_ref = oracle.attention_decode(f64(t["q"][b:b + 1]), f64(t["k"][a:e]), f64(t["v"][a:e]),
                                                 [0, e - a], w.scale)
        assert_fwd_close(o[b:b + 1], lse[:, b:b + 1], o_ref, lse_ref)
