"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or constant with the CUDA library; the two meet only through the
seeded input generator, which holds none of the method's arithmetic.

What it computes is the plain definition of attention, written out with the
N x N score and probability matrices materialised, exactly the data flow the
tiled method is built to avoid:

* "FlashAttention：从 Safe Softmax 到分块计算", section 1 (the formula
  S = QK^T/sqrt(d), P = softmax(S), O = PV and the shapes of each matrix) and
  section 1.1 (one query row: p_ij = e^{s_ij} / sum_t e^{s_it}, o_i = sum_j p_ij v_j).
* the same page, section 2 (safe softmax: subtract the row max before the
  exponential; the result is the same number).
* the same page, section 5.2 (causal mask: s_ij = -inf when j > i, so the
  diagonal stays visible).
* the same page, section 8 (the per-row LogSumExp is the statistic kept for
  the backward pass).
* "企业官网建设流程全解析" (the FlashAttention data-flow notes), section 2.3
  (backward: dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P))); the
  remaining chain-rule steps dQ = scale dS K and dK = scale dS^T Q follow from
  S = scale Q K^T.
* "Attention 算子优化…", section 五 (GQA: consecutive groups of query heads
  share one K/V head) and section 二 (packed variable-length sequences, no
  padding).
* decoding (``attention_decode``): "Attention 算子优化…", section 五 (each
  newly generated token's query attends to the K/V of every earlier token,
  held in the K/V cache: a matrix-vector product per head) and
  "FlashAttention：从 Safe Softmax 到分块计算", section 10 (a decode step with
  one or a few queries calls for a split-K/V strategy such as Flash-Decoding).
  The oracle evaluates the definition directly, with no split; the split
  path's merge is the section 3 rule, which is exact, so the result is the
  same number.

Readings of points the pages leave open (each one is also listed in the design
notes):

* ``scale`` multiplies the raw dot products before masking and softmax; the
  LSE is the natural-log LogSumExp of the *scaled*, masked scores.
* Causal masking uses positions relative to the start of each sequence, and
  key j is visible from query i when j <= i.
* A row with no visible key (only possible for an empty sequence here) gives
  O = 0 and LSE = -inf.
* In a decoding step the new query is the newest token of its sequence and its
  own K/V row is already in the cache, so it sees every cached key: no mask.
* Paged K/V cache ("Attention 算子优化…", section 五, PagedAttention): the cache
  is a pool of fixed-size pages ``[num_pages, page_size, Hkv, d]``; sequence b
  owns logical pages 0, 1, ... whose physical pages are
  ``block_table[b, 0], block_table[b, 1], ...``, and its first ``seqlens[b]``
  logical tokens are its cache.  Table entries past the cache and page
  contents past it are not read.
* Paged prefill (``attention_forward_paged``, the same section's page table
  for a prompt's forward pass): a sequence's queries are its newest tokens and
  its keys are the first ``seqlens_k`` logical tokens of its pages, so when
  the cache holds an earlier part of the sequence the causal mask is aligned
  at the newest token (query i sits at position Lk - Lq + i).
* Layout: tokens-major ``[T, H, d]`` for q/k/v/o and their gradients, ``[Hq, T]``
  for the LSE; sequence s covers tokens ``cu_seqlens[s] .. cu_seqlens[s+1]-1``.

All arithmetic is float64.  Matrix products use numpy's ``@`` (a library
primitive), with no blocking, fusion or reordering beyond the definition.

Parity pins: every function here is checked in ``tests/test_oracle.py``
against the worked examples the pages print, closed forms, invariants and
central finite differences.  The one reading with no pin is that the CUDA
path rounds P to bf16 before the P.V product; the pages are silent on it and it
is bounded only by the stated tolerances.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_decode",
    "attention_decode_paged",
    "attention_forward",
    "attention_forward_paged",
    "attention_forward_rows",
    "attention_backward",
    "tile_counts",
    "tile_counts_closed_form",
    "cu_from_lengths",
]


def cu_from_lengths(lengths) -> np.ndarray:
    """Prefix sums [0, L0, L0+L1, ...] of the sequence lengths (int64)."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def _check_shapes(q, k, v, cu):
    T, Hq, d = q.shape
    Tk, Hkv, dk = k.shape
    if v.shape != k.shape or Tk != T or dk != d:
        raise ValueError("q [T,Hq,d], k and v [T,Hkv,d] expected")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    cu = np.asarray(cu, dtype=np.int64)
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must rise from 0 to T")
    return T, Hq, Hkv, d, cu


def _scores(q_rows, k_rows, scale, causal, q_pos, k_len):
    """Scaled, masked score matrix S for one (sequence, head).

    S[i, j] = scale * <q_i, k_j>; entries with key position > query position
    are -inf under the causal mask (the diagonal stays visible).
    """
    S = scale * (q_rows @ k_rows.T)
    if causal:
        k_pos = np.arange(k_len)
        S = np.where(k_pos[None, :] > np.asarray(q_pos)[:, None], -np.inf, S)
    return S


def _safe_softmax(S):
    """Row-wise safe softmax of S: returns P and the LSE.

    m_i = max_j S_ij; P_ij = exp(S_ij - m_i) / sum_t exp(S_it - m_i);
    LSE_i = m_i + ln sum_t exp(S_it - m_i).  A row that is entirely -inf gives
    P = 0 and LSE = -inf.
    """
    m = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    dead = ~np.isfinite(m)
    m_safe = np.where(dead, 0.0, m)
    E = np.exp(S - m_safe[:, None])
    ell = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(dead[:, None], 0.0, E / np.where(dead, 1.0, ell)[:, None])
        lse = np.where(dead, -np.inf, m_safe + np.log(np.where(dead, 1.0, ell)))
    return P, lse


def attention_forward(q, k, v, cu_seqlens, scale, causal):
    """O and LSE of exact attention over packed sequences (fp64).

    q: [T, Hq, d]; k, v: [T, Hkv, d]; cu_seqlens: [B+1] prefix sums.
    Returns o [T, Hq, d] and lse [Hq, T].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, Hq, Hkv, d, cu = _check_shapes(q, k, v, cu_seqlens)
    group = Hq // Hkv
    o = np.zeros((T, Hq, d), dtype=np.float64)
    lse = np.full((Hq, T), -np.inf, dtype=np.float64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        if L == 0:
            continue
        pos = np.arange(L)
        for h in range(Hq):
            kv = h // group
            S = _scores(q[a:b, h, :], k[a:b, kv, :], scale, causal, pos, L)
            P, lse_rows = _safe_softmax(S)
            o[a:b, h, :] = P @ v[a:b, kv, :]
            lse[h, a:b] = lse_rows
    return o, lse


def attention_forward_rows(q, k, v, cu_seqlens, scale, causal, tokens, heads):
    """O and LSE for selected (token, query head) rows only.

    The same definition as :func:`attention_forward`, evaluated one query row
    at a time, so that single outputs of a full-size problem can be checked.
    Returns o [n, d] and lse [n].
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    heads = np.asarray(heads, dtype=np.int64)
    o = np.zeros((len(tokens), d), dtype=np.float64)
    lse = np.full(len(tokens), -np.inf, dtype=np.float64)
    seq_of = np.searchsorted(cu, tokens, side="right") - 1
    for n in range(len(tokens)):
        s = int(seq_of[n])
        a, b = int(cu[s]), int(cu[s + 1])
        t, h = int(tokens[n]), int(heads[n])
        kv = h // group
        qi = np.asarray(q[t, h, :], dtype=np.float64)[None, :]
        kk = np.asarray(k[a:b, kv, :], dtype=np.float64)
        vv = np.asarray(v[a:b, kv, :], dtype=np.float64)
        S = _scores(qi, kk, scale, causal, [t - a], b - a)
        P, lse_row = _safe_softmax(S)
        o[n] = (P @ vv)[0]
        lse[n] = lse_row[0]
    return o, lse


def attention_decode(q, k, v, cu_seqlens_k, scale):
    """One decoding step: O and LSE for one new query per sequence (fp64).

    q: [B, Hq, d], the query of sequence b's newest token; k, v: [T, Hkv, d],
    the packed K/V cache, sequence b owning rows cu_seqlens_k[b] ..
    cu_seqlens_k[b+1]-1.  Every cached key is visible.  Returns o [B, Hq, d]
    and lse [Hq, B]; a sequence with an empty cache gives O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, d = q.shape
    T, Hkv, dk = k.shape
    cu = np.asarray(cu_seqlens_k, dtype=np.int64)
    if v.shape != k.shape or dk != d or Hq % Hkv != 0:
        raise ValueError("q [B,Hq,d], k and v [T,Hkv,d] with Hq a multiple of Hkv expected")
    if len(cu) != B + 1 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens_k must rise from 0 to T over B + 1 entries")
    group = Hq // Hkv
    o = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.full((Hq, B), -np.inf, dtype=np.float64)
    for b in range(B):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        for h in range(Hq):
            kv = h // group
            S = _scores(q[b, h, :][None, :], k[a:e, kv, :], scale, False, [0], e - a)
            P, lse_row = _safe_softmax(S)
            o[b, h, :] = (P @ v[a:e, kv, :])[0]
            lse[h, b] = lse_row[0]
    return o, lse


def attention_decode_paged(q, k_pages, v_pages, block_table, seqlens, scale):
    """One decoding step over a paged K/V cache (fp64).

    q: [B, Hq, d]; k_pages, v_pages: [num_pages, page_size, Hkv, d];
    block_table: [B, max_pages] physical page of each logical page; seqlens:
    [B] cache lengths.  Gathers each sequence's pages in logical order into a
    packed cache and evaluates :func:`attention_decode` on it.
    """
    k_pages = np.asarray(k_pages, dtype=np.float64)
    v_pages = np.asarray(v_pages, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(seqlens, dtype=np.int64)
    page = k_pages.shape[1]
    ks, vs = [], []
    for b in range(len(lens)):
        L = int(lens[b])
        n = (L + page - 1) // page
        if n > table.shape[1]:
            raise ValueError("block table too short for the cache length")
        rows_k = np.concatenate([k_pages[table[b, j]] for j in range(n)], axis=0)[:L] if n else k_pages[:0, 0]
        rows_v = np.concatenate([v_pages[table[b, j]] for j in range(n)], axis=0)[:L] if n else v_pages[:0, 0]
        ks.append(rows_k)
        vs.append(rows_v)
    k = np.concatenate(ks, axis=0)
    v = np.concatenate(vs, axis=0)
    return attention_decode(q, k, v, cu_from_lengths(lens), scale)


def _gather_pages(pages, table_row, L):
    """The first L logical rows of a sequence whose logical page j is physical
    page table_row[j] of ``pages`` [num_pages, page_size, H, d]."""
    page = pages.shape[1]
    n = (L + page - 1) // page
    if n > len(table_row):
        raise ValueError("block table too short for the cache length")
    if n == 0:
        return pages[:0, 0]
    return np.concatenate([pages[int(table_row[j])] for j in range(n)], axis=0)[:L]


def attention_forward_paged(q, k_pages, v_pages, block_table, cu_seqlens_q, seqlens_k, scale, causal):
    """Prefill over a paged K/V cache: O and LSE of packed queries (fp64).

    q: [Tq, Hq, d]; sequence b's queries are rows cu_seqlens_q[b] ..
    cu_seqlens_q[b+1]-1 (Lq of them), its newest tokens.  Its keys and values
    are the first seqlens_k[b] = Lk logical tokens of its pages in
    k_pages, v_pages [num_pages, page_size, Hkv, d], logical page j being
    physical page block_table[b, j]; when Lk > Lq the first Lk - Lq of them
    are an earlier, cached part of the sequence.  Query i of the sequence is
    the token at position Lk - Lq + i, so under the causal mask it sees keys
    j <= Lk - Lq + i (the mask aligned at the newest token; with Lk = Lq this
    is the ordinary mask).  A row with no visible key gives O = 0 and
    LSE = -inf.  Returns o [Tq, Hq, d] and lse [Hq, Tq].
    """
    q = np.asarray(q, dtype=np.float64)
    k_pages = np.asarray(k_pages, dtype=np.float64)
    v_pages = np.asarray(v_pages, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    lens_k = np.asarray(seqlens_k, dtype=np.int64)
    Tq, Hq, d = q.shape
    Hkv = k_pages.shape[2]
    if Hq % Hkv != 0 or k_pages.shape[3] != d or v_pages.shape != k_pages.shape:
        raise ValueError("q [Tq,Hq,d] and pages [num_pages,page_size,Hkv,d] with Hq a multiple of Hkv expected")
    if cu[0] != 0 or cu[-1] != Tq or np.any(np.diff(cu) < 0) or len(lens_k) != len(cu) - 1:
        raise ValueError("cu_seqlens_q must rise from 0 to Tq over B + 1 entries, seqlens_k have B entries")
    group = Hq // Hkv
    o = np.zeros((Tq, Hq, d), dtype=np.float64)
    lse = np.full((Hq, Tq), -np.inf, dtype=np.float64)
    for b in range(len(lens_k)):
        a, e = int(cu[b]), int(cu[b + 1])
        Lq, Lk = e - a, int(lens_k[b])
        if Lq == 0:
            continue
        K = _gather_pages(k_pages, table[b], Lk)
        V = _gather_pages(v_pages, table[b], Lk)
        q_pos = (Lk - Lq) + np.arange(Lq)
        for h in range(Hq):
            kv = h // group
            S = _scores(q[a:e, h, :], K[:, kv, :], scale, causal, q_pos, Lk)
            P, lse_rows = _safe_softmax(S)
            o[a:e, h, :] = P @ V[:, kv, :]
            lse[h, a:e] = lse_rows
    return o, lse


def attention_backward(q, k, v, do, cu_seqlens, scale, causal, return_rowsum=False):
    """dQ, dK, dV of exact attention for the upstream gradient dO (fp64).

    Per (sequence, query head), with S and P materialised:
      dV  = P^T dO
      dP  = dO V^T
      dS  = P * (dP - rowsum(dP * P))
      dQ  = scale * dS K
      dK  = scale * dS^T Q
    and dK, dV of a K/V head summed over the query heads that share it.
    With ``return_rowsum`` the per-row rowsum(dP * P) is also returned, as
    [Hq, T].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    T, Hq, Hkv, d, cu = _check_shapes(q, k, v, cu_seqlens)
    group = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rowsum = np.zeros((Hq, T), dtype=np.float64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        L = b - a
        if L == 0:
            continue
        pos = np.arange(L)
        for h in range(Hq):
            kv = h // group
            Q, K, V, dO = q[a:b, h, :], k[a:b, kv, :], v[a:b, kv, :], do[a:b, h, :]
            S = _scores(Q, K, scale, causal, pos, L)
            P, _ = _safe_softmax(S)
            dv[a:b, kv, :] += P.T @ dO
            dP = dO @ V.T
            r = (dP * P).sum(axis=1)
            dS = P * (dP - r[:, None])
            dq[a:b, h, :] = scale * (dS @ K)
            dk[a:b, kv, :] += scale * (dS.T @ Q)
            rowsum[h, a:b] = r
    if return_rowsum:
        return dq, dk, dv, rowsum
    return dq, dk, dv


def tile_counts(lengths, causal, Br=128, Bc=128):
    """Number of (query tile, key tile) pairs holding at least one visible score.

    Brute force: for each sequence, enumerate every query tile i and key tile
    j and test whether some (query row r, key column c) in the pair is inside
    the sequence and not masked (c <= r when causal).  This is the work that
    tile skipping leaves ("Attention 算子优化…", section 四: about half of the
    tiles lie entirely under the causal mask and are skipped).  Returns one
    count per sequence (per query head).
    """
    out = []
    for L in lengths:
        L = int(L)
        n = 0
        for i in range(-(-L // Br)):
            r_hi = min(L, (i + 1) * Br) - 1  # last real row of the tile
            for j in range(-(-L // Bc)):
                c_lo = j * Bc  # first column of the tile (always < L here)
                if not causal or c_lo <= r_hi:
                    n += 1
        out.append(n)
    return out


def tile_counts_closed_form(L, causal, B=128):
    """Closed form of :func:`tile_counts` for square tiles Br = Bc = B:
    sum over query tiles i of min(i + 1, ceil(L / B)) when causal, else
    ceil(L / B)^2."""
    n = -(-int(L) // B)
    if not causal:
        return n * n
    return sum(min(i + 1, n) for i in range(n))

