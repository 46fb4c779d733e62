"""Host-side checks of the C ABI: the library loads, exports every entry point
include/fa.h declares, rejects bad arguments before touching a device, and
counts causal tiles exactly as the oracle enumerates them.  No GPU needed."""
import ctypes
import os
import re

import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    from tests.gpu_util import fa_module
    return fa_module()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(fa):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_tile_counts", "fa_stream_status",
            "fa_last_error_string"} <= set(names)
    lib = ctypes.CDLL(fa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(fa.EXPORTS) == set(names)


@pytest.mark.parametrize("lengths", [[1], [127, 128, 129], [4096, 4096], list(
    (6638, 4932, 6735, 1706, 6830, 4356, 1178, 6860)), [0, 5, 300]])
@pytest.mark.parametrize("causal", [False, True])
def test_tile_counts_match_oracle(fa, lengths, causal):
    assert fa.fa_tile_counts(lengths, causal) == oracle.tile_counts(lengths, causal)


def test_workspace_size(fa):
    assert fa.fa_bwd_workspace_size(16, 8192, 64) == 16 * 8192 * 4 + 8192 * 16 * 64 * 4
    assert fa.fa_bwd_workspace_size(0, 10, 64) == 0


def fake(n, align=256):
    """An address that is never dereferenced: argument checks fail first."""
    return n * align


def call_fwd(fa, q=fake(1), k=fake(2), v=fake(3), o=fake(4), lse=fake(5), B=1, Hq=2, Hkv=2, N=128, d=64,
             T=128, scale=0.125, causal=0, cu=None):
    L = fa.lib()
    vp = ctypes.c_void_p
    return L.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, Hq, Hkv, N, d, T, scale, causal, vp(cu), None)


@pytest.mark.parametrize("kw", [
    dict(d=96), dict(d=32), dict(Hq=3, Hkv=2), dict(B=0), dict(N=0), dict(T=100), dict(scale=0.0),
    dict(scale=float("nan")), dict(scale=-1.0), dict(causal=2), dict(q=fake(1) + 8), dict(o=fake(4) + 2),
    dict(lse=fake(5) + 2), dict(k=0), dict(cu=fake(9) + 2),
])
def test_fwd_rejects_bad_arguments_on_host(fa, kw):
    assert call_fwd(fa, **kw) == fa.FA_ERR_INVALID_ARG
    assert fa.lib().fa_last_error_string().decode()


def test_bwd_rejects_bad_arguments_on_host(fa):
    L = fa.lib()
    vp = ctypes.c_void_p
    args = [vp(fake(i + 1)) for i in range(9)]
    # head dimension other than 64 or 128
    rc = L.fa_bwd(*args, 1, 2, 2, 128, 96, 128, 0.1, 1, None, vp(fake(20)), 1 << 30, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    # workspace too small
    rc = L.fa_bwd(*args, 1, 2, 2, 128, 64, 128, 0.1, 1, None, vp(fake(20)), 16, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    # misaligned workspace
    rc = L.fa_bwd(*args, 1, 2, 2, 128, 64, 128, 0.1, 1, None, vp(fake(20) + 16), 1 << 30, None)
    assert rc == fa.FA_ERR_INVALID_ARG


def test_binding_raises_fa_error(fa):
    t = torch.empty(0)
    with pytest.raises(fa.FAError):
        fa._check(call_fwd(fa, d=96))


def test_decode_workspace_size(fa):
    # per (sequence, query head): at most ceil(N / 128) splits of d f32 plus one f32 LSE
    n = 4 * 8 * 32
    assert fa.fa_decode_workspace_size(4, 8, 128, 4096) == n * 128 * 4 + n * 4
    assert fa.fa_decode_workspace_size(1, 1, 64, 1) == 256 + 256
    assert fa.fa_decode_workspace_size(0, 8, 64, 10) == 0


@pytest.mark.parametrize("kw, code", [
    (dict(d=96), "INVALID_ARG"), (dict(Hq=34, Hkv=2), "UNSUPPORTED"), (dict(Hq=3, Hkv=2), "INVALID_ARG"),
    (dict(B=0), "INVALID_ARG"), (dict(T=100), "INVALID_ARG"), (dict(scale=0.0), "INVALID_ARG"),
    (dict(ws_bytes=16), "INVALID_ARG"), (dict(ws=fake(20) + 16), "INVALID_ARG"), (dict(ws=0), "INVALID_ARG"),
    (dict(q=fake(1) + 8), "INVALID_ARG"), (dict(lse=fake(5) + 2), "INVALID_ARG"),
])
def test_decode_rejects_bad_arguments_on_host(fa, kw, code):
    a = dict(q=fake(1), k=fake(2), v=fake(3), o=fake(4), lse=fake(5), B=2, Hq=8, Hkv=2, N=512, d=64, T=1024,
             scale=0.125, cu=None, ws=fake(20), ws_bytes=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    rc = fa.lib().fa_decode(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["o"]), vp(a["lse"]), a["B"], a["Hq"], a["Hkv"],
                            a["N"], a["d"], a["T"], a["scale"], a["cu"], vp(a["ws"]), a["ws_bytes"], None)
    assert rc == getattr(fa, "FA_ERR_" + code)
    assert fa.lib().fa_last_error_string().decode()


@pytest.mark.parametrize("ms", [0, -5, 10001])
def test_selftest_rejects_bad_limits_on_host(fa, ms):
    assert fa.lib().fa_selftest_wait_timeout(ms, None) == fa.FA_ERR_INVALID_ARG
