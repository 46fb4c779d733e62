"""CPU oracle for the FP8 (E4M3) K/V cache (test infrastructure only).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code or table with the CUDA library.

Source: "Attention 算子优化…", section 六 (INT8/FP8 K/V quantisation): the
K/V cache is stored as FP8, E4M3 first of all, with per-token or per-channel
scales; quantisation happens when a block is written back, dequantisation
inside on-chip memory, so HBM only ever holds the compressed form; softmax and
accumulation stay in FP32 and the matrix products in FP16/BF16.

Readings of points the page leaves open (also listed in the design notes):

* Scales are per token and per K/V head: one f32 scale per row of d elements
  of the ``[T, Hkv, d]`` cache, s = max|x| / 448 (448 is the largest finite
  E4M3 value), so the row's largest element maps to +-448.  A row of zeros
  takes s = 1.
* The row is quantised as e4m3(x / s) with round-to-nearest-even and
  saturation to +-448; x / s and s are computed in float32, as the kernel
  does, so that both sides take the rounding decision on the same number.
* E4M3 is the "fn" variant of the format (no infinities, the all-ones code is
  NaN): sign, 4 exponent bits with bias 7, 3 mantissa bits; normal values
  (1 + m/8) 2^(e-7) up to 1.75 * 2^8 = 448, subnormals (m/8) 2^-6.

Parity pins (``tests/test_oracle.py``): the decoding of all 256 codes and the
rounding of a dense sweep of float32 values against torch's ``float8_e4m3fn``
conversion, saturation and ties-to-even by the definition, and the scale rule.
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "e4m3_round", "e4m3_encode", "e4m3_decode", "quantize_rows_fp8", "dequantize_rows_fp8"]

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUBNORMAL_STEP = 2.0 ** -9


def e4m3_round(x):
    """Nearest E4M3 value (ties to even), saturated to +-448; fp64 in and out."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.empty_like(a)
    sub = a < _MIN_NORMAL
    # subnormal range: a fixed step of 2^-9
    out[sub] = np.rint(a[sub] / _SUBNORMAL_STEP) * _SUBNORMAL_STEP
    # normal range: 3 mantissa bits below the leading one, step 2^(E-3)
    an = a[~sub]
    _, e = np.frexp(an)  # an = f * 2^e with f in [0.5, 1): leading bit 2^(e-1)
    step = np.ldexp(1.0, e - 1 - 3)
    out[~sub] = np.rint(an / step) * step
    out = np.minimum(out, E4M3_MAX)
    return np.where(np.isnan(x), np.nan, np.copysign(out, x))


def e4m3_encode(x):
    """Codes (uint8) of e4m3_round(x)."""
    v = e4m3_round(x)
    a = np.abs(v)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = a < _MIN_NORMAL
    code[sub] = np.rint(a[sub] / _SUBNORMAL_STEP).astype(np.uint8)  # exponent field 0
    an = a[~sub]
    _, e = np.frexp(an)
    E = e - 1
    mant = np.rint(an / np.ldexp(1.0, E) * 8 - 8).astype(np.int64)
    code[~sub] = ((E + 7) << 3 | mant).astype(np.uint8)
    return code | sign


def e4m3_decode(code):
    """fp64 values of E4M3 codes (the all-ones exponent-and-mantissa codes are NaN)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * _MIN_NORMAL, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def quantize_rows_fp8(x):
    """Per-row E4M3 quantisation of x [..., d] (bf16-valued).

    Returns (codes uint8 [..., d], scales float32 [...]): s = max|x| / 448 in
    float32 (1 for an all-zero row), codes = e4m3(float32(x) / s)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    q = (x32 / s[..., None]).astype(np.float32)
    return e4m3_encode(q.astype(np.float64)), s


def dequantize_rows_fp8(codes, scales):
    """fp64 values codes * scale (exact)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]
