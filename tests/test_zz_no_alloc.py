"""The allocation-free backward entry point, fa_bwd_noalloc.

Callers that cannot allocate device memory (for example under a runtime whose
memory pool forbids cudaMalloc, or a plugin inside a program that owns all
device memory) use fa_bwd_noalloc, which takes its scratch from an array built
into the library instead of a caller-provided workspace.  These tests call it
through the C ABI and check that it gives the same gradients as fa_bwd with a
workspace, on two calls in a row (the array is shared and keeps the previous
call's contents, so the second call must not depend on them).

Both entry points run the same kernels on the same inputs.  dK and dV are
accumulated inside one thread block in a fixed order, so they must agree bit
for bit; dQ is summed over key tiles by bulk reduce-adds whose order varies
from run to run, so each dQ element may differ by the rounding of that order:
at most one bf16 unit in the last place, plus f32 reduce-order noise for
elements that are tiny against their terms.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_21_gb300.inputs import make_qkv
from tests.gpu_util import fa_module

pytestmark = pytest.mark.gpu


def _setup(lengths, Hq, Hkv, d, causal, seed):
    fa = fa_module()
    dev = torch.device("cuda:0")
    T = sum(lengths)
    t = make_qkv(T, Hq, Hkv, d, seed=seed, with_do=True)
    q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    N = max(lengths)
    o, lse = fa.attention_forward(q, k, v, causal, cu_seqlens=cu, max_seqlen=N)
    return fa, q, k, v, do, o, lse, cu, N, T


def _noalloc(fa, q, k, v, do, o, lse, cu, N, T, causal):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    Hq, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    L = fa.lib()
    vp = ctypes.c_void_p
    rc = L.fa_bwd_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                          vp(do.data_ptr()), vp(lse.data_ptr()), vp(dq.data_ptr()), vp(dk.data_ptr()),
                          vp(dv.data_ptr()), cu.numel() - 1, Hq, Hkv, N, d, T, ctypes.c_float(d ** -0.5),
                          int(causal), vp(cu.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.fa_last_error_string().decode()
    fa.fa_stream_status()
    return dq, dk, dv


def _reference(fa, q, k, v, do, o, lse, cu, N, causal):
    ref = fa.attention_backward(q, k, v, o, lse, do, causal, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    return ref


def _assert_same_gradients(got, ref, what):
    dq, dk, dv = got
    dq_r, dk_r, dv_r = ref
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(x.float()).all(), (what, name)
    # dK and dV: the same kernel, the same order of every sum
    assert torch.equal(dk.view(torch.int16), dk_r.view(torch.int16)), (what, "dk")
    assert torch.equal(dv.view(torch.int16), dv_r.view(torch.int16)), (what, "dv")
    # dQ: one bf16 unit in the last place of the larger of the two values
    a = dq.float().cpu().numpy().astype(np.float64)
    b = dq_r.float().cpu().numpy().astype(np.float64)
    big = np.maximum(np.abs(a), np.abs(b))
    _, e = np.frexp(big)                     # big = m 2^e with m in [0.5, 1)
    ulp = np.ldexp(1.0, e - 8)               # bf16 keeps 8 significant bits
    noise = 1e-4 * float(np.sqrt(np.mean(b * b)))
    bad = np.abs(a - b) > ulp + noise
    assert not bad.any(), (what, "dq", int(bad.sum()), float(np.abs(a - b).max()))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_workspace_backward_twice(cuda_device, causal, d):
    fa, q, k, v, do, o, lse, cu, N, T = _setup([700, 129, 1024, 1], 8, 2, d, causal, seed=31)
    ref = _reference(fa, q, k, v, do, o, lse, cu, N, causal)
    for call in range(2):
        got = _noalloc(fa, q, k, v, do, o, lse, cu, N, T, causal)
        _assert_same_gradients(got, ref, f"call {call}")


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_second_problem_after_larger_one(cuda_device, d):
    """A smaller problem after a larger one: stale scratch must not leak in."""
    fa, q, k, v, do, o, lse, cu, N, T = _setup([2048, 2048], 4, 4, d, True, seed=32)
    _noalloc(fa, q, k, v, do, o, lse, cu, N, T, True)
    fa, q, k, v, do, o, lse, cu, N, T = _setup([300, 77], 4, 4, d, True, seed=33)
    ref = _reference(fa, q, k, v, do, o, lse, cu, N, True)
    got = _noalloc(fa, q, k, v, do, o, lse, cu, N, T, True)
    _assert_same_gradients(got, ref, "after a larger problem")


def test_noalloc_rejects_problems_beyond_the_array(cuda_device):
    fa = fa_module()
    Hq, d = 32, 64
    T = fa.FA_BWD_NOALLOC_SCRATCH_BYTES // (Hq * d * 4) + 1024  # just past the limit
    assert fa.fa_bwd_workspace_size(Hq, T, d) > fa.FA_BWD_NOALLOC_SCRATCH_BYTES
    L = fa.lib()
    vp = ctypes.c_void_p
    fake = [vp(256 * (i + 1)) for i in range(9)]  # never dereferenced: the size check comes first
    rc = L.fa_bwd_noalloc(*fake, 1, Hq, Hq, T, d, T, ctypes.c_float(0.125), 1, None, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    assert "scratch" in L.fa_last_error_string().decode()
