"""GPU parity of decoding over a paged K/V cache against the fp64 oracle.

The pool holds each sequence's pages at a seeded random permutation of its
pages, with noise in unused rows and -1 in unused table entries; the oracle
gathers the same pages through the same table.  Tolerances are the forward's
(bf16 pool) and the FP8 tests' (E4M3 pool).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q8
from exact_attention_21_gb300.inputs import WORKLOADS, make_decode_qkv, make_inputs, make_paged_cache
from tests.gpu_util import FWD_MAX_ABS, FWD_MEAN_ABS, LSE_MAX_ABS, assert_fwd_close, f64, fa_module

pytestmark = pytest.mark.gpu


def paged_case(lengths, Hq, Hkv, d, page, seed):
    t = make_decode_qkv(len(lengths), Hq, int(sum(lengths)), Hkv, d, seed=seed)
    kp, vp, table = make_paged_cache(t["k"], t["v"], lengths, page, seed=seed)
    return t["q"], kp, vp, table


def run(q, kp, vp, table, lengths, page, fp8=False):
    fa = fa_module()
    dev = torch.device("cuda:0")
    qd, kd, vd, td = (x.to(dev).contiguous() for x in (q, kp, vp, table))
    sl = torch.tensor(lengths, dtype=torch.int32, device=dev)
    if fp8:
        k8, ks = fa.kv_quantize_fp8(kd)
        v8, vs = fa.kv_quantize_fp8(vd)
        o, lse = fa.attention_decode_paged(qd, k8, v8, td, sl, page, k_scale=ks, v_scale=vs)
    else:
        o, lse = fa.attention_decode_paged(qd, kd, vd, td, sl, page)
    fa.fa_stream_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_paged(q, kp, vp, table, lengths, page, d, fp8=False):
    Hkv = kp.shape[1]
    k = kp.float().numpy()
    v = vp.float().numpy()
    if fp8:
        k = Q8.dequantize_rows_fp8(*Q8.quantize_rows_fp8(k))
        v = Q8.dequantize_rows_fp8(*Q8.quantize_rows_fp8(v))
    k = k.reshape(-1, page, Hkv, d)
    v = v.reshape(-1, page, Hkv, d)
    return oracle.attention_decode_paged(f64(q), k, v, table.numpy(), lengths, d ** -0.5)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page", [8, 16, 64, 128])
def test_paged_decode(cuda_device, d, page):
    lengths = [5, 1, 300, 128, 129, 0, 640, 77, 2000]
    q, kp, vp, table = paged_case(lengths, 8, 2, d, page, seed=page + d)
    o, lse = run(q, kp, vp, table, lengths, page)
    o_ref, lse_ref = oracle_paged(q, kp, vp, table, lengths, page, d)
    assert_fwd_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page", [16, 128])
def test_paged_decode_fp8(cuda_device, page, d):
    lengths = [5, 1, 300, 129, 0, 640, 2000]
    q, kp, vp, table = paged_case(lengths, 32, 4, d, page, seed=page + d)
    o, lse = run(q, kp, vp, table, lengths, page, fp8=True)
    o_ref, lse_ref = oracle_paged(q, kp, vp, table, lengths, page, d, fp8=True)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all() and err.max() <= FWD_MAX_ABS
    assert err.mean() <= FWD_MEAN_ABS + 2.0 ** -9 * np.abs(o_ref).mean()
    fin = np.isfinite(lse_ref)
    assert np.abs(lse[fin] - lse_ref[fin]).max() <= LSE_MAX_ABS


def test_paged_decode_rejects_bad_table_entries_and_lengths(cuda_device):
    """An entry inside a cache that is not a page of the pool, or a length
    above max_pages * page_size, is reported by fa_stream_status; the kernels
    read page 0 instead, so nothing outside the pool is touched."""
    fa = fa_module()
    lengths = [40, 40]
    q, kp, vp, table = paged_case(lengths, 4, 1, 128, 16, seed=3)
    bad = table.clone()
    bad[1, 1] = kp.shape[0] // 16 + 5
    for tab, lens in ((bad, lengths), (table, [40, 16 * table.shape[1] + 1])):
        dev = torch.device("cuda:0")
        with pytest.raises(fa.FAError) as e:
            o, lse = fa.attention_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), tab.to(dev),
                                               torch.tensor(lens, dtype=torch.int32, device=dev), 16)
            fa.fa_stream_status()
        assert e.value.code == fa.FA_ERR_INVALID_ARG
    # the context stays usable
    o, lse = run(q, kp, vp, table, lengths, 16)
    assert np.isfinite(o).all()


def test_paged_decode_workload(cuda_device):
    """Full-size paged workload, checked on three whole sequences."""
    w = WORKLOADS["decode_paged16_b64_hq64_hkv8_n4096_d128"]
    t = make_inputs(w)
    o, lse = run(t["q"], t["k_pages"], t["v_pages"], t["block_table"], w.seq_lengths, w.page_size)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    cu = oracle.cu_from_lengths(w.seq_lengths)
    for b in [0, 40, w.B - 1]:
        a, e = int(cu[b]), int(cu[b + 1])
        o_ref, lse_ref = oracle.attention_decode(f64(t["q"][b:b + 1]), f64(t["k"][a:e]), f64(t["v"][a:e]),
                                                 [0, e - a], w.scale)
        assert_fwd_close(o[b:b + 1], lse[:, b:b + 1], o_ref, lse_ref)
