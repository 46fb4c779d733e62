"""GPU parity of the prefill over a paged K/V cache (fa_fwd_paged).

Each sequence's keys and values live in pages scattered over a pool (seeded
random placement, noise in unused rows, -1 in unused table entries).  Cases:
no cached prefix (Lk = Lq), a cached prefix (Lk > Lq, mask aligned at the
newest token), fewer keys than queries under the mask (rows with no visible
key), empty query chunks, page sizes 8-128, GQA, both head dimensions.  The
outputs are compared element by element with the oracle's paged prefill at the
forward bars; with Lk = Lq they must also equal the contiguous packed forward
bit for bit (the same arithmetic, only the loads differ).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs, make_paged_cache, make_qkv
from tests.gpu_util import assert_fwd_close, f64, fa_module

pytestmark = pytest.mark.gpu


def _case(Lq, Lk, Hq, Hkv, d, page, seed):
    tq = make_qkv(sum(Lq), Hq, Hkv, d, seed=seed)
    tk = make_qkv(sum(Lk), Hq, Hkv, d, seed=seed + 1)
    kp, vp, table = make_paged_cache(tk["k"], tk["v"], Lk, page, seed=seed)
    return tq["q"], tk["k"], tk["v"], kp, vp, table


def _run(q, kp, vp, table, Lq, Lk, page, causal, scale):
    fa = fa_module()
    dev = torch.device("cuda:0")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(Lq)]), dtype=torch.int32, device=dev)
    lk = torch.tensor(Lk, dtype=torch.int32, device=dev)
    o, lse = fa.attention_forward_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), cu, lk, max(max(Lq), 1),
                                        page, causal, scale=scale)
    fa.fa_stream_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(q, kp, vp, table, Lq, Lk, page, causal, scale):
    Hkv, d = kp.shape[1], kp.shape[2]
    shape = (kp.shape[0] // page, page, Hkv, d)
    return oracle.attention_forward_paged(f64(q), f64(kp).reshape(shape), f64(vp).reshape(shape),
                                          table.numpy(), oracle.cu_from_lengths(Lq), Lk, scale, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("page", [8, 16, 64, 128])
def test_paged_prefill_with_cached_prefix(cuda_device, d, causal, page):
    """Chunks of new queries after cached prefixes of various lengths (tile
    edges, ragged tails, a one-query chunk, an empty chunk), GQA 4/2."""
    Lq = [300, 1, 128, 0, 77, 129, 256]
    Lk = [300, 700, 383, 50, 77, 260, 511]
    q, k, v, kp, vp, table = _case(Lq, Lk, 4, 2, d, page, seed=60 + page)
    o, lse = _run(q, kp, vp, table, Lq, Lk, page, causal, d ** -0.5)
    o_ref, lse_ref = _oracle(q, kp, vp, table, Lq, Lk, page, causal, d ** -0.5)
    assert_fwd_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_paged_prefill_rows_without_keys(cuda_device, d):
    """Causal with fewer keys than queries: the first Lq - Lk rows see no key
    and give O = 0, LSE = -inf; the rest match the oracle."""
    Lq, Lk = [200, 140], [70, 140]
    q, k, v, kp, vp, table = _case(Lq, Lk, 2, 1, d, 16, seed=70)
    o, lse = _run(q, kp, vp, table, Lq, Lk, 16, True, d ** -0.5)
    o_ref, lse_ref = _oracle(q, kp, vp, table, Lq, Lk, 16, True, d ** -0.5)
    assert np.all(o[:130] == 0.0) and np.all(np.isneginf(lse[:, :130]))
    assert np.all(np.isneginf(lse_ref[:, :130]))
    assert_fwd_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page", [8, 32])
def test_paged_prefill_equals_packed_forward_bitwise(cuda_device, d, page):
    """Lk = Lq: the same tiles in the same order as the contiguous packed
    forward, so the same bits."""
    fa = fa_module()
    L = [5, 300, 128, 129, 640, 77]
    q, k, v, kp, vp, table = _case(L, L, 8, 2, d, page, seed=80)
    o, lse = _run(q, kp, vp, table, L, L, page, True, d ** -0.5)
    dev = torch.device("cuda:0")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(L)]), dtype=torch.int32, device=dev)
    # the same keys and values, contiguous
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o2, lse2 = fa.attention_forward(qd, kd, vd, True, cu_seqlens=cu, max_seqlen=max(L))
    fa.fa_stream_status()
    assert np.array_equal(o, o2.float().cpu().numpy())
    assert np.array_equal(lse, lse2.cpu().numpy())


def test_paged_prefill_bad_table_entry_is_reported(cuda_device):
    fa = fa_module()
    Lq, Lk = [100], [100]
    q, k, v, kp, vp, table = _case(Lq, Lk, 1, 1, 64, 16, seed=90)
    table[0, 2] = 10_000  # not a page of the pool
    with pytest.raises(fa.FAError) as ei:
        _run(q, kp, vp, table, Lq, Lk, 16, True, 0.125)
    assert ei.value.code == fa.FA_ERR_INVALID_ARG
    fa.fa_stream_status()  # cleared


def test_paged_prefill_workload_sampled_rows(cuda_device):
    """The packed workload's sequences and heads (Hq32/Hkv8, d128, causal) with
    K/V in 16-token pages: every output finite and bounded, sampled rows
    against the oracle, and bitwise equality with the packed forward."""
    fa = fa_module()
    w = WORKLOADS["fwd_paged16_varlen8_hq32_hkv8_d128_causal"]
    t = make_inputs(w)
    dev = torch.device("cuda:0")
    L = w.seq_lengths
    o, lse = _run(t["q"], t["k_pages"], t["v_pages"], t["block_table"], L, L, w.page_size, True, w.scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(L)]), dtype=torch.int32, device=dev)
    o2, lse2 = fa.attention_forward(t["q"].to(dev), t["k"].to(dev), t["v"].to(dev), True, cu_seqlens=cu,
                                    max_seqlen=w.N)
    fa.fa_stream_status()
    assert np.array_equal(o, o2.float().cpu().numpy())
    r = np.random.default_rng(7)
    toks = r.integers(0, w.T, 128)
    heads = r.integers(0, w.Hq, 128)
    cu_np = oracle.cu_from_lengths(L)
    o_ref, lse_ref = oracle.attention_forward_rows(f64(t["q"]), f64(t["k"]), f64(t["v"]), cu_np, w.scale, True,
                                                   toks, heads)
    err = np.abs(o[toks, heads] - o_ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse[heads, toks] - lse_ref).max() <= 1e-3
