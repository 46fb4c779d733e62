"""CPU model of the E4M3-term number format the FP8 decoding step uses.

The tensor-core decoding step over an E4M3 cache multiplies 8-bit operands
only: the query and the probabilities are each carried as a sum of three E4M3
numbers (t1 = e4m3(y), t2 = e4m3(y - t1), t3 = e4m3(y - t1 - t2)).  For the
probabilities the kernel takes w = p * s_v * 2^(6 + 126 - E), E the largest
biased exponent of the V scales seen so far, with the running max allowed to
lag by at most 2 (log2 units), so that w < 256 and the weights that carry O
stay in E4M3's normal range.

These tests run that recipe in numpy, with E4M3 rounding taken from the
oracle's pinned ``e4m3_round``, and check what the design relies on: the
three-term sum of w is within 2^-12 |w| of it for w >= 4 and within 2^-10
(half E4M3's subnormal step) below, the weights never reach E4M3's largest
value, and O computed from the term sums (the lazy reference, the exponent E
and the rescales included) is within 2^-9 max|O| of the exact attention over
the same dequantised cache: no coarser than the bf16 P of the bf16-cache
kernel, and far inside the 1e-2 / 1e-3 bars of the GPU tests.  They do not
run the kernel: the GPU parity tests do.
"""
import numpy as np
import pytest

from oracle.quant import E4M3_MAX, dequantize_rows_fp8, e4m3_round, quantize_rows_fp8

SLACK = 2.0       # lag of the running max, log2 units
P_SCALE_LOG2 = 6  # the weights carry p s_v 2^(6 + 126 - E)


def terms(y, n=3):
    """The n E4M3 terms of y, and their sum."""
    out, r = [], np.asarray(y, dtype=np.float64)
    for _ in range(n):
        t = e4m3_round(r)
        out.append(t)
        r = r - t
    return out, sum(out)


def test_three_terms_hold_a_weight_to_2_pow_minus_12_relative_or_2_pow_minus_10():
    rng = np.random.default_rng(1)
    y = np.exp2(rng.uniform(-8.0, 8.0, size=40000)) * rng.choice([-1, 1], size=40000)
    _, s = terms(y)
    assert np.all(np.abs(s - y) <= np.maximum(2.0 ** -12 * np.abs(y), 2.0 ** -10))
    big = np.abs(y) >= 4.0
    assert np.max(np.abs(s - y)[big] / np.abs(y)[big]) <= 2.0 ** -12
    _, s2 = terms(y, 2)
    # two terms only reach about 2^-8 on large weights: the reason for the third
    assert np.max(np.abs(s2 - y)[big] / np.abs(y)[big]) > 2.0 ** -10


def biased_exponent(s):
    return np.frexp(s)[1] + 126  # s = f 2^e, f in [0.5, 1): biased exponent e - 1 + 127


def model_decode(q, kd, vc, vs, scale, tile=128):
    """O of one query head over one cache, the kernel's way: scores of the
    dequantised keys (the S^T side is modelled exactly), probabilities against
    a lazily moved reference, weights w split into three E4M3 terms, and V
    taken as the E4M3 codes with the scales folded into w."""
    c = scale * np.log2(np.e)
    x = (kd @ q) * c
    m, E, l, o, wmax = -np.inf, 0, 0.0, np.zeros(vc.shape[1]), 0.0
    for t0 in range(0, len(x), tile):
        xs, sv = x[t0:t0 + tile], vs[t0:t0 + tile]
        ei = biased_exponent(sv)
        alpha = beta = 1.0
        if xs.max() > m + SLACK or ei.max() > E:
            if xs.max() > m + SLACK:
                alpha = np.exp2(m - xs.max()) if np.isfinite(m) else 0.0
                m = xs.max()
            if ei.max() > E:
                beta = np.exp2(E - ei.max())
                E = int(ei.max())
        p = np.exp2(xs - m)
        l = l * alpha + p.sum()
        svs = sv * np.exp2(P_SCALE_LOG2 + 126 - E)
        w = p * svs
        wmax = max(wmax, w.max())
        _, wsum = terms(w)
        o = o * alpha * beta + wsum @ vc[t0:t0 + tile]
    return o * np.exp2(E - 126 - P_SCALE_LOG2) / l, wmax


@pytest.mark.parametrize("n, q_mult, v_mult", [(1, 1, 1), (129, 1, 1), (1000, 1, 1), (4096, 1, 1), (4096, 4, 1),
                                               (4096, 1, 1e-4), (4096, 1, 1e4), (3000, 8, 1e-3)])
def test_model_decode_matches_exact_attention_over_the_dequantised_cache(n, q_mult, v_mult):
    rng = np.random.default_rng(n + int(q_mult))
    d = 128
    q = rng.standard_normal(d) * q_mult
    k = rng.standard_normal((n, d)).astype(np.float32)
    v = (rng.standard_normal((n, d)) * v_mult).astype(np.float32)
    kd = dequantize_rows_fp8(*quantize_rows_fp8(k))
    vcodes, vs = quantize_rows_fp8(v)
    vc = dequantize_rows_fp8(vcodes, np.ones_like(vs))  # the codes' values
    vd = dequantize_rows_fp8(vcodes, vs)
    s = (kd @ q) * d ** -0.5
    pe = np.exp(s - s.max())
    exact = pe @ vd / pe.sum()
    got, wmax = model_decode(q, kd, vc, vs.astype(np.float64), d ** -0.5)
    assert wmax < 256.0 < E4M3_MAX  # no weight saturates
    err = np.abs(got - exact)
    assert err.max() <= 2.0 ** -9 * np.abs(exact).max(), (err.max(), np.abs(exact).max())
