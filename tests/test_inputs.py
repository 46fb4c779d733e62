"""CPU checks of the seeded input generators and of the workload accounting
that bench.py divides by (no GPU, no attention arithmetic).

The algorithmic FLOP count is checked against a count of the visible
(query, key) pairs, each costing 4 d FLOPs (2 d for the score, 2 d for its
share of P V); the decoding byte count against the tensors a step reads and
writes; the paged cache against the packed cache it was cut from.
"""
import numpy as np
import pytest
import torch

from exact_attention_21_gb300.inputs import (VARLEN_LENGTHS, WORKLOADS, Workload, cu_seqlens_of, make_decode_qkv,
                                             make_inputs, make_paged_cache, make_qkv)


def visible_pairs(L, causal):
    """Number of (query, key) pairs the softmax covers in one sequence."""
    return L * (L + 1) // 2 if causal else L * L


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if not w.decode])
def test_fwd_flops_count_the_visible_pairs(name):
    w = WORKLOADS[name]
    exact = sum(4 * w.d * visible_pairs(L, w.causal) for L in w.seq_lengths) * w.Hq
    if w.causal:
        # the causal count is the usual convention, half of the full square;
        # the diagonal adds L/2 pairs per sequence on top of it
        assert w.fwd_flops() == pytest.approx(exact, rel=1.0 / min(w.seq_lengths))
        assert w.fwd_flops() < exact
    else:
        assert w.fwd_flops() == exact
    assert w.bwd_flops() == 2.5 * w.fwd_flops()


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.decode])
def test_decode_bytes_are_the_tensors_a_step_touches(name):
    w = WORKLOADS[name]
    t = make_inputs(w) if w.T * w.Hkv * w.d <= (1 << 26) else None
    kv_elems = w.T * w.Hkv * w.d
    if w.fp8:
        cache = 2 * kv_elems * 1 + 2 * w.T * w.Hkv * 4  # E4M3 codes + an f32 scale per token and head
    else:
        cache = 2 * kv_elems * 2
    q_and_o = 2 * w.B * w.Hq * w.d * 2
    lse = w.B * w.Hq * 4
    assert w.decode_bytes() == cache + q_and_o + lse
    if t is not None:
        assert t["k"].numel() == kv_elems and t["q"].shape == (w.B, w.Hq, w.d)


def test_workload_shapes_and_lengths():
    w = WORKLOADS["fwd_varlen8_hq32_hkv8_d128_causal"]
    assert w.seq_lengths == list(VARLEN_LENGTHS) and w.T == sum(VARLEN_LENGTHS) == 39235
    assert w.N == max(VARLEN_LENGTHS) and w.Hq % w.Hkv == 0
    assert all(512 <= L <= 8192 for L in VARLEN_LENGTHS)
    b = WORKLOADS["fwdbwd_b2_h16_n4096_d64_causal"]
    assert (b.B, b.Hq, b.N, b.d, b.causal, b.backward) == (2, 16, 4096, 64, True, True)
    assert b.scale == pytest.approx(64 ** -0.5)
    assert cu_seqlens_of([3, 0, 5]).tolist() == [0, 3, 3, 8]


def test_generators_are_seeded_and_bf16():
    a, b, c = make_qkv(40, 4, 2, 64, seed=3, with_do=True), make_qkv(40, 4, 2, 64, seed=3, with_do=True), \
        make_qkv(40, 4, 2, 64, seed=4, with_do=True)
    for n in ("q", "k", "v", "do"):
        assert a[n].dtype == torch.bfloat16
        assert torch.equal(a[n], b[n])
        assert not torch.equal(a[n], c[n])
    assert a["q"].shape == (40, 4, 64) and a["k"].shape == (40, 2, 64)
    d = make_decode_qkv(3, 8, 50, 2, 128, seed=1)
    assert d["q"].shape == (3, 8, 128) and d["v"].shape == (50, 2, 128)
    # N(0, 1) draws: moments of a few thousand samples
    x = a["q"].float()
    assert abs(x.mean().item()) < 0.1 and abs(x.std().item() - 1.0) < 0.1


@pytest.mark.parametrize("page", [8, 16, 128])
def test_paged_cache_gathers_back_to_the_packed_cache(page):
    lengths = [5, 0, 300, 128, 129, 17]
    t = make_decode_qkv(len(lengths), 4, sum(lengths), 2, 64, seed=page)
    kp, vp, table = make_paged_cache(t["k"], t["v"], lengths, page, seed=page)
    used = table[table >= 0].tolist()
    assert len(used) == len(set(used))  # no page is shared
    assert all(0 <= pg < kp.shape[0] // page for pg in used)
    start = 0
    for b, L in enumerate(lengths):
        npg = (L + page - 1) // page
        assert (table[b, :npg] >= 0).all() and (table[b, npg:] == -1).all()
        for j in range(L):
            row = int(table[b, j // page]) * page + j % page
            assert torch.equal(kp[row], t["k"][start + j]) and torch.equal(vp[row], t["v"][start + j])
        start += L


def test_paged_workload_inputs_match_their_packed_cache():
    w = Workload("paged_probe", 3, 8, 2, 300, 64, False, (300, 1, 129), False, True, False, 16)
    t = make_inputs(w)
    assert t["seqlens"].tolist() == [300, 1, 129]
    kp, table = t["k_pages"], t["block_table"]
    cu = t["cu_seqlens"].tolist()
    for b, L in enumerate(w.seq_lengths):
        rows = [int(table[b, j // 16]) * 16 + j % 16 for j in range(L)]
        assert torch.equal(kp[rows], t["k"][cu[b]:cu[b + 1]])
    assert np.all(np.diff(cu) == np.array(w.seq_lengths))
