"""GPU parity of the FP8 (E4M3) K/V cache path against the CPU oracle.

Quantisation is integer work decided by float32 arithmetic on both sides:
codes and scales must match the oracle's bit for bit.  A decoding step over
the E4M3 cache is compared with the fp64 oracle's attention over the oracle's
own dequantised cache (codes x scales), with the forward's tolerances plus
one allowance: a dequantised value (code x f32 scale) is in general not a
bf16 number, so storing O in bf16 costs up to 2^-9 |O| per element even when
O is a single cached V row (caches of one token give |O| of order 1).  The
mean bound is therefore 1e-3 + 2^-9 mean|O_ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q8
from exact_attention_21_gb300.inputs import WORKLOADS, make_decode_qkv, make_inputs
from tests.gpu_util import FWD_MAX_ABS, FWD_MEAN_ABS, LSE_MAX_ABS, f64, fa_module

pytestmark = pytest.mark.gpu


def gpu_quantize(x):
    fa = fa_module()
    x8, s = fa.kv_quantize_fp8(x.to("cuda:0").contiguous())
    fa.fa_stream_status()
    return x8.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_matches_oracle_bit_for_bit(cuda_device, d):
    g = torch.Generator().manual_seed(d)
    x = torch.randn(700, 3, d, generator=g)
    x[5, 1] = 0.0                      # all-zero row: scale 1, codes 0
    x[6, 0] *= 1e-4                    # tiny values: subnormal codes
    x[7, 2] *= 3e4                     # large values
    x[8, 1, :] = 0.5                   # constant row: every code +448
    x[9, 0, ::2] = -x[9, 0, 1::2]      # sign pattern
    xb = x.to(torch.bfloat16)
    codes, scales = gpu_quantize(xb)
    ref_codes, ref_scales = Q8.quantize_rows_fp8(xb.float().numpy())
    np.testing.assert_array_equal(scales.view(np.uint32), ref_scales.view(np.uint32))
    np.testing.assert_array_equal(codes, ref_codes)


def run_decode_fp8(t, lengths=None, N=None):
    fa = fa_module()
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev).contiguous() for n in ("q", "k", "v"))
    k8, ks = fa.kv_quantize_fp8(k)
    v8, vs = fa.kv_quantize_fp8(v)
    if lengths is None:
        cu = None
    else:
        N = max(max(lengths), 1)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o, lse = fa.attention_decode_fp8(q, k8, v8, ks, vs, cu_seqlens_k=cu, max_seqlen_k=N)
    fa.fa_stream_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_decode_fp8(t, cu, scale):
    """fp64 attention over the oracle's own dequantised cache."""
    k = Q8.dequantize_rows_fp8(*Q8.quantize_rows_fp8(t["k"].float().numpy()))
    v = Q8.dequantize_rows_fp8(*Q8.quantize_rows_fp8(t["v"].float().numpy()))
    return oracle.attention_decode(f64(t["q"]), k, v, cu, scale)


def assert_fp8_close(o, lse, o_ref, lse_ref):
    assert np.isfinite(o).all(), "NaN/Inf in O"
    finite = np.isfinite(lse_ref)
    assert np.isfinite(lse[finite]).all(), "NaN/Inf in LSE"
    err = np.abs(o - o_ref)
    assert err.max() <= FWD_MAX_ABS, f"max |dO| = {err.max():.3e}"
    assert err.mean() <= FWD_MEAN_ABS + 2.0 ** -9 * np.abs(o_ref).mean(), f"mean |dO| = {err.mean():.3e}"
    if finite.any():
        assert np.abs(lse[finite] - lse_ref[finite]).max() <= LSE_MAX_ABS
    return err.max(), err.mean()


def check(B, Hq, Hkv, lengths, batched=False, seed=0, d=128):
    T = int(sum(lengths))
    t = make_decode_qkv(B, Hq, T, Hkv, d, seed=seed)
    o, lse = run_decode_fp8(t, lengths=None if batched else lengths, N=lengths[0] if batched else None)
    o_ref, lse_ref = oracle_decode_fp8(t, oracle.cu_from_lengths(lengths), d ** -0.5)
    return assert_fp8_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (16, 2), (64, 8)])
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_decode_fp8_d64_head_pairs(cuda_device, heads, N):
    """d = 64 over an E4M3 cache: adjacent K/V heads paired into 128-byte rows,
    each softmax warpgroup using its own head's per-token scales."""
    check(3, heads[0], heads[1], [N] * 3, batched=True, seed=N + heads[0], d=64)


def test_decode_fp8_d64_packed_ragged_and_many_items(cuda_device):
    check(9, 8, 2, [5, 1, 300, 128, 129, 0, 640, 77, 2000], seed=6, d=64)
    lengths = [int(x) for x in np.random.default_rng(33).integers(0, 700, size=160)]
    check(len(lengths), 8, 2, lengths, seed=33, d=64)


def test_decode_fp8_d64_unpaired_is_unsupported(cuda_device):
    """Odd Hkv (or a group above 8) at d = 64: no E4M3 kernel, a clear error."""
    fa = fa_module()
    t = make_decode_qkv(2, 3, 200, 3, 64, seed=8)
    with pytest.raises(fa.FAError) as e:
        run_decode_fp8(t, lengths=[100, 100])
    assert e.value.code == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("N", [1, 129, 1000])
def test_decode_fp8_batched(cuda_device, N):
    check(3, 8, 2, [N] * 3, batched=True, seed=N)


def test_decode_fp8_packed_ragged_with_empty_caches(cuda_device):
    check(9, 8, 2, [5, 1, 300, 128, 129, 0, 640, 77, 2000], seed=5)


@pytest.mark.parametrize("heads", [(4, 4), (24, 8), (32, 2)])
def test_decode_fp8_gqa_groups(cuda_device, heads):
    check(2, heads[0], heads[1], [700, 1500], seed=sum(heads))


@pytest.mark.parametrize("heads", [(8, 2), (32, 2)])
def test_decode_fp8_many_items_per_cta(cuda_device, heads):
    """A dozen items per CTA of mixed and empty lengths: the per-token scales
    are copied ahead across items (and loaded directly for the tiles the
    ring could not reach), and the scale exponent restarts with each item."""
    lengths = [int(x) for x in np.random.default_rng(32).integers(0, 700, size=160)]
    check(len(lengths), heads[0], heads[1], lengths, seed=32)


def test_decode_fp8_long_cache_many_splits(cuda_device):
    check(1, 4, 1, [20000], batched=True, seed=7)


def test_decode_fp8_close_to_the_bf16_cache(cuda_device):
    """Sanity of scale: the E4M3 cache changes O by about the quantisation
    step (2^-4 relative per element), far less than O's own size."""
    fa = fa_module()
    t = make_decode_qkv(4, 16, 4 * 2048, 4, 128, seed=13)
    o8, _ = run_decode_fp8(t, N=2048)
    dev = torch.device("cuda:0")
    o16, _ = fa.attention_decode(*(t[n].to(dev) for n in ("q", "k", "v")), max_seqlen_k=2048)
    diff = np.abs(o8 - o16.float().cpu().numpy())
    assert diff.mean() < 0.05 * np.abs(o8).mean()


def test_decode_fp8_workload(cuda_device):
    """Full-size FP8 decoding workload, checked on three whole sequences."""
    w = WORKLOADS["decode_fp8_b64_hq64_hkv8_n4096_d128"]
    t = make_inputs(w)
    o, lse = run_decode_fp8(t, N=w.N)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    for b in [0, 31, w.B - 1]:
        a, e = b * w.N, (b + 1) * w.N
        sub = {"q": t["q"][b:b + 1], "k": t["k"][a:e], "v": t["v"][a:e]}
        o_ref, lse_ref = oracle_decode_fp8(sub, [0, w.N], w.scale)
        assert_fp8_close(o[b:b + 1], lse[:, b:b + 1], o_ref, lse_ref)
