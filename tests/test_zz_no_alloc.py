"""The allocation-free backward entry point, fa_bwd_noalloc.

Callers that cannot allocate device memory (for example under a runtime whose
memory pool forbids cudaMalloc, or a plugin inside a program that owns all
device memory) use fa_bwd_noalloc, which takes its scratch from an array built
into the library instead of a caller-provided workspace.  These tests call it
through the C ABI and check that it gives the same gradients as fa_bwd with a
workspace, on two calls in a row (the array is shared and keeps the previous
call's contents, so the second call must not depend on them).

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_21_gb300.inputs import make_qkv
from tests.gpu_util import BWD_REL_FRO, fa_module, rel_fro

pytestmark = pytest.mark.gpu


def _setup(lengths, Hq, Hkv, causal, seed):
    fa = fa_module()
    dev = torch.device("cuda:0")
    T = sum(lengths)
    t = make_qkv(T, Hq, Hkv, 64, seed=seed, with_do=True)
    q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    N = max(lengths)
    o, lse = fa.attention_forward(q, k, v, causal, cu_seqlens=cu, max_seqlen=N)
    return fa, q, k, v, do, o, lse, cu, N, T


def _noalloc(fa, q, k, v, do, o, lse, cu, N, T, causal):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    Hq, Hkv = q.shape[1], k.shape[1]
    L = fa.lib()
    vp = ctypes.c_void_p
    rc = L.fa_bwd_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                          vp(do.data_ptr()), vp(lse.data_ptr()), vp(dq.data_ptr()), vp(dk.data_ptr()),
                          vp(dv.data_ptr()), cu.numel() - 1, Hq, Hkv, N, 64, T, 0.125, int(causal),
                          vp(cu.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.fa_last_error_string().decode()
    fa.fa_stream_status()
    return [x.float().cpu().numpy() for x in (dq, dk, dv)]


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_workspace_backward_twice(cuda_device, causal):
    fa, q, k, v, do, o, lse, cu, N, T = _setup([700, 129, 1024, 1], 8, 2, causal, seed=31)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    ref = [x.float().cpu().numpy() for x in ref]
    for call in range(2):
        got = _noalloc(fa, q, k, v, do, o, lse, cu, N, T, causal)
        for name, x, r in zip(("dq", "dk", "dv"), got, ref):
            assert np.isfinite(x).all(), (call, name)
            assert rel_fro(x, r) <= BWD_REL_FRO, (call, name, rel_fro(x, r))


def test_noalloc_second_problem_after_larger_one(cuda_device):
    """A smaller problem after a larger one: stale scratch must not leak in."""
    fa, q, k, v, do, o, lse, cu, N, T = _setup([2048, 2048], 4, 4, True, seed=32)
    _noalloc(fa, q, k, v, do, o, lse, cu, N, T, True)
    fa, q, k, v, do, o, lse, cu, N, T = _setup([300, 77], 4, 4, True, seed=33)
    ref = fa.attention_backward(q, k, v, o, lse, do, True, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    got = _noalloc(fa, q, k, v, do, o, lse, cu, N, T, True)
    for x, r in zip(got, ref):
        assert rel_fro(x, r.float().cpu().numpy()) <= BWD_REL_FRO


def test_noalloc_rejects_problems_beyond_the_array(cuda_device):
    fa = fa_module()
    Hq, d = 32, 64
    T = fa.FA_BWD_NOALLOC_SCRATCH_BYTES // (Hq * d * 4) + 1024  # just past the limit
    assert fa.fa_bwd_workspace_size(Hq, T, d) > fa.FA_BWD_NOALLOC_SCRATCH_BYTES
    L = fa.lib()
    vp = ctypes.c_void_p
    fake = [vp(256 * (i + 1)) for i in range(9)]  # never dereferenced: the size check comes first
    rc = L.fa_bwd_noalloc(*fake, 1, Hq, Hq, T, d, T, 0.125, 1, None, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    assert "scratch" in L.fa_last_error_string().decode()
