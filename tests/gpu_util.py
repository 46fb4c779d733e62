"""Helpers shared by the GPU parity tests: run the CUDA path through the
C ABI binding and compare with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle

FWD_MAX_ABS = 1e-2   # max |dO| against the fp64 oracle
FWD_MEAN_ABS = 1e-3  # mean |dO|
LSE_MAX_ABS = 1e-3   # max |dLSE|
BWD_REL_FRO = 2e-2   # ||dX - dX_ref||_F / ||dX_ref||_F for X in {Q, K, V}


def fa_module():
    import exact_attention_21_gb300.fa as fa
    import exact_attention_21_gb300.build as b
    import os
    if not os.path.exists(fa.LIB_PATH):
        b.build()
    return fa


def f64(t):
    return t.to(torch.float64).numpy()


def run_fwd(q, k, v, causal, lengths=None, N=None, scale=None):
    """q, k, v: CPU bf16 [T, H, d].  Returns o (f32 numpy), lse (numpy)."""
    fa = fa_module()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev).contiguous() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    if lengths is None:
        N = N or T
        B = T // N
        cu = None
    else:
        B = len(lengths)
        N = max(max(lengths), 1)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    fa.fa_fwd(qd, kd, vd, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu)
    fa.fa_stream_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def cu_of(T, lengths=None, N=None):
    if lengths is not None:
        return oracle.cu_from_lengths(lengths)
    N = N or T
    return np.arange(0, T + 1, N, dtype=np.int64)


def assert_fwd_close(o, lse, o_ref, lse_ref, rows=None):
    assert np.isfinite(o).all(), "NaN/Inf in O"
    finite = np.isfinite(lse_ref)
    assert np.isfinite(lse[finite]).all(), "NaN/Inf in LSE"
    err = np.abs(o - o_ref)
    assert err.max() <= FWD_MAX_ABS, f"max |dO| = {err.max():.3e}"
    assert err.mean() <= FWD_MEAN_ABS, f"mean |dO| = {err.mean():.3e}"
    lerr = np.abs(lse[finite] - lse_ref[finite])
    if lerr.size:
        assert lerr.max() <= LSE_MAX_ABS, f"max |dLSE| = {lerr.max():.3e}"
    return err.max(), err.mean(), (lerr.max() if lerr.size else 0.0)


def rel_fro(x, ref):
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30))
