"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only names the workloads and
draws their inputs, so both the CUDA path's tests and the CPU oracle can be fed
from the same bytes.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws float32 standard normals in the order q, k, v, dO, each shaped
``[T, H, d]`` (token-major, head dimension innermost), and each is rounded to
bfloat16 (round to nearest even).  ``scale`` is 1/sqrt(d).  Packed
variable-length workloads list their sequence lengths literally; they were drawn
once as ``torch.randint(512, 8193, (8,))`` from a CPU generator seeded 0 and are
frozen here so that no torch version can change them.

Decoding workloads (``decode=True``) have one new query token per sequence:
the generator draws q shaped ``[B, Hq, d]`` and then k, v shaped
``[T, Hkv, d]`` (the K/V cache, T = the summed cache lengths), each rounded to
bfloat16 as above.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_decode_qkv", "make_inputs", "make_paged_cache", "make_qkv"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int  # sequence length (batched) or the longest sequence (packed)
    d: int
    causal: bool
    lengths: tuple = field(default=())  # packed sequences; empty = batched
    backward: bool = False
    decode: bool = False  # one new query per sequence against a K/V cache of the lengths above
    fp8: bool = False     # decoding over an E4M3 cache with per-token f32 scales
    page_size: int = 0    # K/V in a paged cache with pages of this many tokens (0: contiguous)

    @property
    def seq_lengths(self) -> list:
        return list(self.lengths) if self.lengths else [self.N] * self.B

    @property
    def T(self) -> int:
        return sum(self.seq_lengths)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def varlen(self) -> bool:
        return bool(self.lengths)

    def kv_cache_bytes(self) -> int:
        """Bytes of the K and V caches a decoding step reads (bf16, or E4M3
        codes plus one f32 scale per token and K/V head)."""
        if self.fp8:
            return 2 * self.T * self.Hkv * (self.d + 4)
        return 2 * self.T * self.Hkv * self.d * 2

    def decode_bytes(self) -> int:
        """Algorithmic bytes of one decoding step: the K/V caches read once,
        q and o (bf16) and the LSE (f32)."""
        return self.kv_cache_bytes() + 2 * self.B * self.Hq * self.d * 2 + self.B * self.Hq * 4

    def decode_flops(self) -> float:
        """Algorithmic FLOPs of one decoding step: 4 L d per (sequence, query head)."""
        return sum(4.0 * L * self.d for L in self.seq_lengths) * self.Hq

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs: 4 L^2 d per (sequence, query head),
        halved under the causal mask."""
        f = sum(4.0 * L * L * self.d for L in self.seq_lengths) * self.Hq
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """Algorithmic backward FLOPs: 2.5 x the forward count."""
        return 2.5 * self.fwd_flops()


VARLEN_LENGTHS = (6638, 4932, 6735, 1706, 6830, 4356, 1178, 6860)

WORKLOADS = {
    "fwd_b1_h1_n256_d64": Workload("fwd_b1_h1_n256_d64", 1, 1, 1, 256, 64, False),
    "fwd_b4_h16_n2048_d64": Workload("fwd_b4_h16_n2048_d64", 4, 16, 16, 2048, 64, False),
    "fwd_b2_h32_n4096_d128_causal": Workload(
        "fwd_b2_h32_n4096_d128_causal", 2, 32, 32, 4096, 128, True),
    "fwd_varlen8_hq32_hkv8_d128_causal": Workload(
        "fwd_varlen8_hq32_hkv8_d128_causal", 8, 32, 8, max(VARLEN_LENGTHS), 128, True,
        VARLEN_LENGTHS),
    "fwdbwd_b2_h16_n4096_d64_causal": Workload(
        "fwdbwd_b2_h16_n4096_d64_causal", 2, 16, 16, 4096, 64, True, (), True),
    "fwdbwd_b2_h32_n4096_d128_causal": Workload(
        "fwdbwd_b2_h32_n4096_d128_causal", 2, 32, 32, 4096, 128, True, (), True),
    # 64 sequences with 4096 cached tokens each, 64 query heads sharing 8 K/V
    # heads (the grouping the GQA section names for Llama-2 70B), d = 128: one
    # step reads 1.07 GB of K/V cache.
    "decode_b64_hq64_hkv8_n4096_d128": Workload(
        "decode_b64_hq64_hkv8_n4096_d128", 64, 64, 8, 4096, 128, False, (), False, True),
    # the same step at head dimension 64 (0.54 GB of cache)
    "decode_b64_hq64_hkv8_n4096_d64": Workload(
        "decode_b64_hq64_hkv8_n4096_d64", 64, 64, 8, 4096, 64, False, (), False, True),
    # the same step over an E4M3 cache (per-token scales)
    "decode_fp8_b64_hq64_hkv8_n4096_d128": Workload(
        "decode_fp8_b64_hq64_hkv8_n4096_d128", 64, 64, 8, 4096, 128, False, (), False, True, True),
    # the d = 64 step over an E4M3 cache
    "decode_fp8_b64_hq64_hkv8_n4096_d64": Workload(
        "decode_fp8_b64_hq64_hkv8_n4096_d64", 64, 64, 8, 4096, 64, False, (), False, True, True),
    # the same step with the cache in 16-token pages scattered over a pool
    "decode_paged16_b64_hq64_hkv8_n4096_d128": Workload(
        "decode_paged16_b64_hq64_hkv8_n4096_d128", 64, 64, 8, 4096, 128, False, (), False, True, False, 16),
    # prefill of the packed workload's sequences and heads with K/V in 16-token
    # pages scattered over a pool (no cached prefix: keys = queries)
    "fwd_paged16_varlen8_hq32_hkv8_d128_causal": Workload(
        "fwd_paged16_varlen8_hq32_hkv8_d128_causal", 8, 32, 8, max(VARLEN_LENGTHS), 128, True, VARLEN_LENGTHS,
        False, False, False, 16),
    # the packed workload's sequences and heads, one new token each
    "decode_varlen8_hq32_hkv8_d128": Workload(
        "decode_varlen8_hq32_hkv8_d128", 8, 32, 8, max(VARLEN_LENGTHS), 128, False, VARLEN_LENGTHS, False,
        True),
}


def make_qkv(T, Hq, Hkv, d, seed=0, with_do=False, q_mult=1.0):
    """Draw q [T,Hq,d], k, v [T,Hkv,d] (and dO [T,Hq,d]) as bf16 CPU tensors.

    ``q_mult`` multiplies the float32 draw of q before rounding (stress cases
    with a wide score range)."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, Hq, d, generator=g)
    k = torch.randn(T, Hkv, d, generator=g)
    v = torch.randn(T, Hkv, d, generator=g)
    out = {
        "q": (q * q_mult).to(torch.bfloat16),
        "k": k.to(torch.bfloat16),
        "v": v.to(torch.bfloat16),
    }
    if with_do:
        out["do"] = torch.randn(T, Hq, d, generator=g).to(torch.bfloat16)
    return out


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_decode_qkv(B, Hq, T, Hkv, d, seed=0):
    """Draw q [B,Hq,d] (one new query per sequence) and the K/V cache k, v
    [T,Hkv,d] as bf16 CPU tensors."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(T, Hkv, d, generator=g)
    v = torch.randn(T, Hkv, d, generator=g)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}


def make_paged_cache(k, v, lengths, page_size, seed=0, spare_pages=3):
    """Lays a packed cache k, v [T, Hkv, d] out as a page pool.

    Each sequence's rows are cut into pages of ``page_size`` tokens, and the
    pages (plus ``spare_pages`` unused ones) are placed at a seeded random
    permutation of the pool's pages.  Unused pool rows are filled with seeded
    noise.  Returns (k_pages, v_pages [num_pages * page_size, Hkv, d],
    block_table int32 [B, max_pages] with -1 in unused entries)."""
    g = torch.Generator().manual_seed(seed + 7919)
    T, Hkv, d = k.shape
    npg = [(int(L) + page_size - 1) // page_size for L in lengths]
    total = sum(npg) + spare_pages
    max_pages = max(npg + [1])
    perm = torch.randperm(total, generator=g)
    kp = torch.randn(total * page_size, Hkv, d, generator=g).to(k.dtype)
    vp = torch.randn(total * page_size, Hkv, d, generator=g).to(v.dtype)
    table = torch.full((len(lengths), max_pages), -1, dtype=torch.int32)
    nxt, start = 0, 0
    for b, L in enumerate(lengths):
        L = int(L)
        for j in range(npg[b]):
            pg = int(perm[nxt])
            nxt += 1
            table[b, j] = pg
            a, e = start + j * page_size, min(start + (j + 1) * page_size, start + L)
            kp[pg * page_size:pg * page_size + e - a] = k[a:e]
            vp[pg * page_size:pg * page_size + e - a] = v[a:e]
        start += L
    return kp, vp, table


def make_inputs(w: Workload, seed=0, with_do=None):
    """Inputs of workload ``w`` on the CPU: q, k, v (, do) bf16 and cu_seqlens int32
    (decoding workloads: q [B,Hq,d], the K/V cache and its offsets)."""
    if w.decode:
        t = make_decode_qkv(w.B, w.Hq, w.T, w.Hkv, w.d, seed=seed)
        t["cu_seqlens"] = cu_seqlens_of(w.seq_lengths)
        if w.page_size:
            t["k_pages"], t["v_pages"], t["block_table"] = make_paged_cache(t["k"], t["v"], w.seq_lengths,
                                                                           w.page_size, seed=seed)
            t["seqlens"] = torch.tensor(w.seq_lengths, dtype=torch.int32)
        return t
    if with_do is None:
        with_do = w.backward
    t = make_qkv(w.T, w.Hq, w.Hkv, w.d, seed=seed, with_do=with_do)
    t["cu_seqlens"] = cu_seqlens_of(w.seq_lengths)
    if w.page_size:
        # prefill over a paged cache: the same k, v laid out in pages
        t["k_pages"], t["v_pages"], t["block_table"] = make_paged_cache(t["k"], t["v"], w.seq_lengths, w.page_size,
                                                                       seed=seed)
        t["seqlens"] = torch.tensor(w.seq_lengths, dtype=torch.int32)
    return t
