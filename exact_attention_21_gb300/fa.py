"""ctypes binding of libfa.so: the same entry points as include/fa.h.

Argument marshalling only: tensors are passed as device pointers with the
current torch CUDA stream, and a non-zero status becomes an ``FAError``.
Every step of the computation runs in the library's CUDA kernels; there is no
other implementation behind these functions, and loading fails loudly when
the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED_DEVICE = 2
FA_ERR_LAUNCH = 3
FA_ERR_TIMEOUT = 4
FA_ERR_UNSUPPORTED = 5

EXPORTS = ("fa_fwd", "fa_fwd_counted", "fa_fwd_paged", "fa_bwd", "fa_bwd_counted", "fa_bwd_deterministic", "fa_bwd_noalloc", "fa_bwd_workspace_size", "fa_decode", "fa_decode_fp8",
           "fa_decode_paged", "fa_decode_paged_fp8", "fa_decode_workspace_size", "fa_kv_quantize_fp8",
           "fa_selftest_wait_timeout", "fa_tile_counts", "fa_stream_status", "fa_last_error_string",
           "fa_launch_count")


class FAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"fa error {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """Loads libfa.so once; raises if it is missing (build it first)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run exact_attention_21_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp]
        L.fa_fwd.restype = i32
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp,
                             ctypes.c_size_t, vp]
        L.fa_bwd.restype = i32
        L.fa_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32, i32, i32,
                                   i32, vp]
        L.fa_fwd_paged.restype = i32
        L.fa_fwd_counted.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp, vp]
        L.fa_fwd_counted.restype = i32
        L.fa_bwd_counted.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp,
                                     vp, ctypes.c_size_t, vp, vp]
        L.fa_bwd_counted.restype = i32
        L.fa_bwd_deterministic.argtypes = list(L.fa_bwd.argtypes)
        L.fa_bwd_deterministic.restype = i32
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, i32,
                                     vp, vp]
        L.fa_bwd_noalloc.restype = i32
        L.fa_bwd_workspace_size.argtypes = [i32, i64, i32]
        L.fa_bwd_workspace_size.restype = ctypes.c_size_t
        L.fa_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, vp, vp, ctypes.c_size_t, vp]
        L.fa_decode.restype = i32
        L.fa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i64, f32, vp, vp,
                                    ctypes.c_size_t, vp]
        L.fa_decode_fp8.restype = i32
        L.fa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp,
                                      ctypes.c_size_t, vp]
        L.fa_decode_paged.restype = i32
        L.fa_decode_paged_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                          vp, ctypes.c_size_t, vp]
        L.fa_decode_paged_fp8.restype = i32
        L.fa_kv_quantize_fp8.argtypes = [vp, vp, vp, i64, i32, vp]
        L.fa_kv_quantize_fp8.restype = i32
        L.fa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        L.fa_decode_workspace_size.restype = ctypes.c_size_t
        L.fa_tile_counts.argtypes = [i32, ctypes.POINTER(ctypes.c_int), i32, ctypes.POINTER(ctypes.c_longlong)]
        L.fa_tile_counts.restype = i32
        L.fa_selftest_wait_timeout.argtypes = [i32, vp]
        L.fa_selftest_wait_timeout.restype = i32
        L.fa_stream_status.argtypes = [vp]
        L.fa_stream_status.restype = i32
        L.fa_last_error_string.argtypes = []
        L.fa_last_error_string.restype = ctypes.c_char_p
        L.fa_launch_count.argtypes = []
        L.fa_launch_count.restype = ctypes.c_ulonglong
        _lib = L
    return _lib


def _check(rc):
    if rc != FA_OK:
        raise FAError(rc, lib().fa_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens=None, stream=None):
    """Forward pass into caller-allocated ``o`` [T,Hq,d] bf16 and ``lse`` [Hq,T] f32."""
    _check(lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, T, float(scale),
                        int(causal), _ptr(cu_seqlens), _stream(stream)))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace,
           stream=None):
    """Backward pass into caller-allocated ``dq``, ``dk``, ``dv`` (bf16)."""
    _check(lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, Hq, Hkv, N, d, T, float(scale), int(causal), _ptr(cu_seqlens), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream)))


def fa_fwd_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seqlens_k, o, lse, max_seqlen_q, page_size, scale,
                 causal, stream=None):
    """Prefill over a paged K/V cache into caller-allocated ``o`` [Tq,Hq,d] and
    ``lse`` [Hq,Tq]; the pools are [num_pages * page_size, Hkv, d]."""
    Tq, Hq, d = q.shape
    Hkv = k_pages.shape[1]
    B, max_pages = block_table.shape
    num_pages = k_pages.shape[0] // page_size
    _check(lib().fa_fwd_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(cu_seqlens_q),
                              _ptr(seqlens_k), _ptr(o), _ptr(lse), B, Hq, Hkv, max_seqlen_q, d, Tq, float(scale),
                              int(causal), page_size, num_pages, max_pages, _stream(stream)))


def attention_forward_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seqlens_k, max_seqlen_q, page_size,
                            causal, scale=None, stream=None):
    """Allocates O and LSE and runs :func:`fa_fwd_paged`."""
    Tq, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device)
    fa_fwd_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seqlens_k, o, lse, max_seqlen_q, page_size,
                 d ** -0.5 if scale is None else scale, causal, stream)
    return o, lse


def fa_fwd_counted(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, tile_counts, stream=None):
    """:func:`fa_fwd`, and the (query tile, key tile) pairs the kernel computed
    per sequence (summed over query heads) into ``tile_counts`` (int64 [B])."""
    _check(lib().fa_fwd_counted(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, T, float(scale),
                                int(causal), _ptr(cu_seqlens), _ptr(tile_counts), _stream(stream)))


def fa_bwd_counted(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace,
                   tile_counts, stream=None):
    """:func:`fa_bwd`, and the (key tile, query tile) pairs the gradient kernel
    computed per sequence (summed over query heads) into ``tile_counts``."""
    _check(lib().fa_bwd_counted(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, Hq, Hkv, N, d, T, float(scale), int(causal), _ptr(cu_seqlens),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(tile_counts),
                                _stream(stream)))


def fa_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens,
                         workspace, stream=None):
    """:func:`fa_bwd` with run-to-run bitwise reproducible results."""
    _check(lib().fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                      _ptr(dv), B, Hq, Hkv, N, d, T, float(scale), int(causal), _ptr(cu_seqlens),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens=None,
                   stream=None):
    """Backward pass without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in scratch array is used
    instead (at most FA_BWD_NOALLOC_SCRATCH_BYTES; calls share it, so calls
    that overlap on the GPU must be ordered by the caller)."""
    _check(lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, Hq, Hkv, N, d, T, float(scale), int(causal), _ptr(cu_seqlens),
                                _stream(stream)))


FA_BWD_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def fa_bwd_workspace_size(Hq, T, d):
    return int(lib().fa_bwd_workspace_size(Hq, T, d))


def fa_decode(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, workspace, stream=None):
    """One decoding step into caller-allocated ``o`` [B,Hq,d] bf16 and ``lse`` [Hq,B] f32."""
    _check(lib().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, T, float(scale),
                           _ptr(cu_seqlens_k), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream)))


def fa_decode_fp8(q, k8, v8, k_scale, v_scale, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, workspace,
                  stream=None):
    """One decoding step over an E4M3 cache (uint8 codes, f32 per-token scales)."""
    _check(lib().fa_decode_fp8(_ptr(q), _ptr(k8), _ptr(v8), _ptr(k_scale), _ptr(v_scale), _ptr(o), _ptr(lse), B, Hq,
                               Hkv, N, d, T, float(scale), _ptr(cu_seqlens_k), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)))


def fa_decode_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, page_size, scale, workspace, stream=None):
    """One decoding step over a paged cache: pools [num_pages * page_size, Hkv, d], table [B, max_pages]."""
    B, Hq, d = q.shape
    Hkv = k_pages.shape[1]
    _check(lib().fa_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens), _ptr(o),
                                 _ptr(lse), B, Hq, Hkv, d, page_size, k_pages.shape[0] // page_size,
                                 block_table.shape[1], float(scale), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def fa_decode_paged_fp8(q, k8_pages, v8_pages, k_scale, v_scale, block_table, seqlens, o, lse, page_size, scale,
                        workspace, stream=None):
    """:func:`fa_decode_paged` over an E4M3 pool with per-token scales [num_pages * page_size, Hkv]."""
    B, Hq, d = q.shape
    Hkv = k8_pages.shape[1]
    _check(lib().fa_decode_paged_fp8(_ptr(q), _ptr(k8_pages), _ptr(v8_pages), _ptr(k_scale), _ptr(v_scale),
                                     _ptr(block_table), _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, page_size,
                                     k8_pages.shape[0] // page_size, block_table.shape[1], float(scale),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def attention_decode_paged(q, k_pages, v_pages, block_table, seqlens, page_size, scale=None, k_scale=None,
                           v_scale=None, stream=None):
    """Allocates o, lse and the workspace and runs a decoding step over a paged
    cache (bf16 pools, or E4M3 pools when k_scale and v_scale are given)."""
    B, Hq, d = q.shape
    if scale is None:
        scale = d ** -0.5
    ws = torch.empty(fa_decode_workspace_size(B, Hq, d, block_table.shape[1] * page_size), dtype=torch.uint8,
                     device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, B, dtype=torch.float32, device=q.device)
    if k_scale is None:
        fa_decode_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, page_size, scale, ws, stream)
    else:
        fa_decode_paged_fp8(q, k_pages, v_pages, k_scale, v_scale, block_table, seqlens, o, lse, page_size, scale,
                            ws, stream)
    return o, lse


def fa_kv_quantize_fp8(x, x8, scale, stream=None):
    """Quantises bf16 rows x [..., d] into E4M3 codes x8 (uint8, same shape) and scales [...] (f32)."""
    d = x.shape[-1]
    _check(lib().fa_kv_quantize_fp8(_ptr(x), _ptr(x8), _ptr(scale), x.numel() // d, d, _stream(stream)))


def kv_quantize_fp8(x, stream=None):
    """Allocates and returns (codes uint8 [..., d], scales f32 [...]) for bf16 rows x."""
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    fa_kv_quantize_fp8(x, x8, scale, stream)
    return x8, scale


def fa_decode_workspace_size(B, Hq, d, max_seqlen_k):
    return int(lib().fa_decode_workspace_size(B, Hq, d, max_seqlen_k))


def fa_tile_counts(lengths, causal):
    n = len(lengths)
    arr = (ctypes.c_int * max(n, 1))(*[int(x) for x in lengths])
    out = (ctypes.c_longlong * max(n, 1))()
    _check(lib().fa_tile_counts(n, arr, int(causal), out))
    return [int(out[i]) for i in range(n)]


def fa_selftest_wait_timeout(limit_ms, stream=None):
    """Runs the bounded-wait self-test (a wait that nothing completes)."""
    _check(lib().fa_selftest_wait_timeout(int(limit_ms), _stream(stream)))


def fa_stream_status(stream=None):
    """Synchronises the stream and raises on a latched device-side error."""
    _check(lib().fa_stream_status(_stream(stream)))


def fa_launch_count():
    """Kernels the library has launched in this process so far."""
    return int(lib().fa_launch_count())


# ---------------------------------------------------------------- conveniences

def attention_forward(q, k, v, causal, scale=None, cu_seqlens=None, max_seqlen=None, stream=None):
    """Allocates o and lse with torch and calls :func:`fa_fwd`.

    q [T,Hq,d], k/v [T,Hkv,d] bf16 CUDA tensors; batched mode takes
    ``q.shape[0] == B * N`` with ``max_seqlen = N`` (default: one sequence).
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    if cu_seqlens is None:
        N = max_seqlen or T
        B = T // N
    else:
        B = cu_seqlens.numel() - 1
        N = max_seqlen
    o = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, stream)
    return o, lse


def attention_decode(q, k, v, scale=None, cu_seqlens_k=None, max_seqlen_k=None, workspace=None, stream=None):
    """Allocates o, lse (and the workspace if not given) and calls :func:`fa_decode`.

    q [B,Hq,d]: one new query per sequence; k/v [T,Hkv,d]: the K/V cache,
    batched (``T == B * max_seqlen_k``) or packed by ``cu_seqlens_k``.
    """
    B, Hq, d = q.shape
    T, Hkv, _ = k.shape
    if scale is None:
        scale = d ** -0.5
    if cu_seqlens_k is None:
        N = max_seqlen_k or T // B
    else:
        N = max_seqlen_k
    if workspace is None:
        workspace = torch.empty(fa_decode_workspace_size(B, Hq, d, N), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, B, dtype=torch.float32, device=q.device)
    fa_decode(q, k, v, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, workspace, stream)
    return o, lse


def attention_decode_fp8(q, k8, v8, k_scale, v_scale, scale=None, cu_seqlens_k=None, max_seqlen_k=None,
                         workspace=None, stream=None):
    """:func:`attention_decode` over an E4M3 cache (see :func:`kv_quantize_fp8`)."""
    B, Hq, d = q.shape
    T, Hkv, _ = k8.shape
    if scale is None:
        scale = d ** -0.5
    N = max_seqlen_k if (cu_seqlens_k is not None or max_seqlen_k) else T // B
    if workspace is None:
        workspace = torch.empty(fa_decode_workspace_size(B, Hq, d, N), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty(Hq, B, dtype=torch.float32, device=q.device)
    fa_decode_fp8(q, k8, v8, k_scale, v_scale, o, lse, B, Hq, Hkv, N, d, T, scale, cu_seqlens_k, workspace, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dout, causal, scale=None, cu_seqlens=None, max_seqlen=None,
                       workspace=None, stream=None, deterministic=False):
    """Allocates dq, dk, dv (and the workspace if not given) and calls :func:`fa_bwd`."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    if cu_seqlens is None:
        N = max_seqlen or T
        B = T // N
    else:
        B = cu_seqlens.numel() - 1
        N = max_seqlen
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(Hq, T, d), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    call = fa_bwd_deterministic if deterministic else fa_bwd
    call(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, T, scale, causal, cu_seqlens, workspace, stream)
    return dq, dk, dv
