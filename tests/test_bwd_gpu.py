"""GPU parity of the backward kernels against the fp64 oracle's gradients.

The CUDA backward consumes the CUDA forward's O and LSE, as a user would; the
oracle differentiates the exact attention of the same bf16 inputs.  The bar is
a relative Frobenius error <= 2e-2 on each of dQ, dK, dV.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import WORKLOADS, make_inputs, make_qkv
from tests.gpu_util import BWD_REL_FRO, assert_fwd_close, cu_of, f64, fa_module, rel_fro

pytestmark = pytest.mark.gpu


def run_fwd_bwd(t, causal, lengths=None, N=None, with_fwd=False):
    fa = fa_module()
    dev = torch.device("cuda:0")
    q, k, v, do = (t[n].to(dev).contiguous() for n in ("q", "k", "v", "do"))
    T, Hq, d = q.shape
    if lengths is None:
        N = N or T
        cu = None
    else:
        N = max(max(lengths), 1)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o, lse = fa.attention_forward(q, k, v, causal, cu_seqlens=cu, max_seqlen=N)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    grads = [x.float().cpu().numpy() for x in (dq, dk, dv)]
    if with_fwd:
        return grads, o.float().cpu().numpy(), lse.cpu().numpy()
    return grads


def check(t, causal, lengths=None, N=None):
    got = run_fwd_bwd(t, causal, lengths, N)
    T, _, d = t["q"].shape
    ref = oracle.attention_backward(f64(t["q"]), f64(t["k"]), f64(t["v"]), f64(t["do"]), cu_of(T, lengths, N),
                                    d ** -0.5, causal)
    errs = {}
    for name, x, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(x).all(), f"NaN/Inf in {name}"
        if np.linalg.norm(r) == 0.0:
            # one visible key per row (N = 1): P = 1 exactly and dS = 0, so
            # the exact gradient is zero and only rounding noise may remain
            assert np.abs(x).max() <= 1e-4, (name, np.abs(x).max())
            errs[name] = 0.0
        else:
            errs[name] = rel_fro(x, r)
    assert max(errs.values()) <= BWD_REL_FRO, errs
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 127, 128, 129, 300, 512])
def test_bwd_single_sequence(cuda_device, causal, N, d):
    check(make_qkv(N, 2, 2, d, seed=10, with_do=True), causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_batched_gqa(cuda_device, causal, d):
    check(make_qkv(3 * 384, 8, 2, d, seed=11, with_do=True), causal, N=384)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_packed_ragged(cuda_device, causal, d):
    lengths = [5, 1, 300, 128, 129, 0, 640, 77]
    check(make_qkv(sum(lengths), 4, 1, d, seed=12, with_do=True), causal, lengths=lengths)


@pytest.mark.parametrize("name", ["fwdbwd_b2_h16_n4096_d64_causal", "fwdbwd_b2_h32_n4096_d128_causal"])
def test_bwd_workload(cuda_device, name):
    """Full-size forward+backward workloads.  B2 H16 N4096 d64 causal: the
    forward's O and LSE and the backward's dQ, dK, dV of every one of the 32
    (sequence, head) slices against the oracle on that slice.  The d = 128
    shape (64 slices): eight slices spread over both sequences and the heads.
    Both: sum_j dK_j = 0 over the whole output."""
    w = WORKLOADS[name]
    t = make_inputs(w)
    (dq, dk, dv), o, lse = run_fwd_bwd(t, w.causal, N=w.N, with_fwd=True)
    for x in (dq, dk, dv, o):
        assert np.isfinite(x).all()
    # sum_j dK_j = 0 per (sequence, head): dS rows sum to zero
    for b in range(w.B):
        sl = slice(b * w.N, (b + 1) * w.N)
        col = np.abs(dk[sl].sum(axis=0)).max()
        assert col <= 2e-2 * np.abs(dk[sl]).sum(axis=0).max() + 1e-3, col
    if w.d == 64:
        pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    else:
        pairs = [(0, 0), (0, 9), (0, 22), (0, 31), (1, 3), (1, 14), (1, 25), (1, 30)]
    err_sum, n_el = 0.0, 0
    for b, h in pairs:
        sl = slice(b * w.N, (b + 1) * w.N)
        sub = {n: f64(t[n][sl, h:h + 1]) for n in ("q", "k", "v", "do")}
        o_ref, lse_ref = oracle.attention_forward(sub["q"], sub["k"], sub["v"], [0, w.N], w.scale, w.causal)
        e_max, e_mean, l_max = assert_fwd_close(o[sl, h:h + 1], lse[h:h + 1, sl], o_ref, lse_ref)
        err_sum += e_mean * o_ref.size
        n_el += o_ref.size
        ref = oracle.attention_backward(sub["q"], sub["k"], sub["v"], sub["do"], [0, w.N], w.scale, w.causal)
        for gname, x, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            e = rel_fro(x[sl, h:h + 1], r)
            assert e <= BWD_REL_FRO, (b, h, gname, e)
    assert err_sum / n_el <= 1e-3


# ---------------------------------------------------------------- deterministic backward

def run_bwd_det(t, causal, lengths=None, N=None, repeats=1):
    fa = fa_module()
    dev = torch.device("cuda:0")
    q, k, v, do = (t[n].to(dev).contiguous() for n in ("q", "k", "v", "do"))
    T = q.shape[0]
    if lengths is None:
        N = N or T
        cu = None
    else:
        N = max(max(lengths), 1)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
    o, lse = fa.attention_forward(q, k, v, causal, cu_seqlens=cu, max_seqlen=N)
    outs = []
    for _ in range(repeats):
        outs.append(fa.attention_backward(q, k, v, o, lse, do, causal, cu_seqlens=cu, max_seqlen=N,
                                          deterministic=True))
    fast = fa.attention_backward(q, k, v, o, lse, do, causal, cu_seqlens=cu, max_seqlen=N)
    fa.fa_stream_status()
    return outs, fast


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", ["single", "gqa", "packed"])
def test_bwd_deterministic_parity(cuda_device, d, causal, case):
    if case == "single":
        t, kw, T = make_qkv(300, 2, 2, d, seed=20, with_do=True), {}, 300
    elif case == "gqa":
        t, kw, T = make_qkv(3 * 384, 8, 2, d, seed=21, with_do=True), {"N": 384}, 3 * 384
    else:
        lengths = [5, 1, 300, 128, 129, 0, 640, 77]
        t, kw, T = make_qkv(sum(lengths), 4, 1, d, seed=22, with_do=True), {"lengths": lengths}, sum(lengths)
    outs, _ = run_bwd_det(t, causal, **kw)
    got = [x.float().cpu().numpy() for x in outs[0]]
    ref = oracle.attention_backward(f64(t["q"]), f64(t["k"]), f64(t["v"]), f64(t["do"]),
                                    cu_of(T, kw.get("lengths"), kw.get("N")), d ** -0.5, causal)
    for name, x, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(x).all(), name
        assert rel_fro(x, r) <= BWD_REL_FRO, (name, rel_fro(x, r))


@pytest.mark.parametrize("name", ["fwdbwd_b2_h16_n4096_d64_causal", "fwdbwd_b2_h32_n4096_d128_causal"])
def test_bwd_deterministic_is_bitwise_reproducible(cuda_device, name):
    """Three runs give identical bits; dK and dV also equal the fast
    backward's bit for bit (the same kernel without its dQ part), and dQ
    agrees with the fast backward's to its rounding."""
    w = WORKLOADS[name]
    t = make_inputs(w)
    outs, fast = run_bwd_det(t, w.causal, N=w.N, repeats=3)
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), fast[1].view(torch.int16))
    assert torch.equal(outs[0][2].view(torch.int16), fast[2].view(torch.int16))
    dq_d, dq_f = outs[0][0].float(), fast[0].float()
    assert ((dq_d - dq_f).norm() / dq_f.norm()).item() <= 1e-2
