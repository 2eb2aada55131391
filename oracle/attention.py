"""fp64 CPU oracle for the FlashAttention-2 forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path; the only common input is ``fa_inputs`` (seeded
random draws, no attention arithmetic).

What the method computes
------------------------
Page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与 TiledMMA",
section 先看全局 (first display equation): for one query tile,
S = Q K^T, P = softmax(S), O = P V.  With the softmax scale, the causal mask
and the per-row log-sum-exp that the production FA2 kernel also returns
(section 与官方 FA2 比较时，先对齐契约, the contract table row "输出"), the
plain definition for batch b, head h and query row i < S is

    N_i      = { j : j < S }                      (non-causal)
             = { j : j <= i }                     (causal)
    z_ij     = scale * sum_d Q[b,i,h,d] K[b,j,h,d]
    M_i      = max_{j in N_i} z_ij
    P_ij     = exp(z_ij - M_i) / sum_{j in N_i} exp(z_ij - M_i)
    O[b,i,h] = sum_{j in N_i} P_ij V[b,j,h]
    LSE[b,h,i] = M_i + ln sum_{j in N_i} exp(z_ij - M_i)

``attention_reference`` writes exactly that, in fp64, from the 16-bit input
values decoded exactly.  Nothing is blocked, fused or reordered beyond
computing a few query rows at a time to bound memory.

``online_softmax_attention`` is a second, independent fp64 implementation
that follows the pages' recurrence (section 沿 C fragment 做 Online Softmax,
the three display equations there, and section 教学配置 for the state m_i,
l_i, o~_i): it walks the keys in tiles and keeps a running max, a running
sum and an unnormalised output, rescaling both by alpha = exp(m_old - m_new)
whenever the max moves.  It is used to pin the algebra the GPU kernel relies
on (including the lazy variant that keeps a stale max until it grows by more
than a threshold) against the plain definition.

Readings where the pages are silent
-----------------------------------
* causal: key j is visible to query i iff j <= i (square self-attention).
* scale multiplies Q K^T before the softmax; LSE is the natural log of the
  sum of exp of the *scaled* logits.
* layout: [B, S, H, D] for Q, K, V, O; LSE is [B, H, S].
* padded keys (j >= S) do not exist in the definition; every row has at least
  one visible key (j = 0), so no row is empty.
* grouped K/V heads (not on the pages; the production extension listed with
  the contract): K and V may have H_kv heads with H_kv dividing H; query head
  h then uses K/V head h // (H / H_kv), consecutive query heads sharing one
  K/V head (H_kv = 1: one K/V head for all).
* variable-length batches (not on the pages; "变长序列" is listed with the
  production FA2's other needs): sequences packed along the token axis,
  Q [total, H, D], K and V [total, H_kv, D], offsets cu[0..B] with cu[0] = 0;
  sequence b is rows cu[b] .. cu[b+1]-1 and attends only within itself (the
  causal mask counts positions from the sequence start); LSE is [H, total].
* local (sliding-window) attention (not on the pages beyond "causal/local
  mask" among the production needs): a window (left, right) keeps key j for
  query i iff i - left <= j <= i + right, a negative bound meaning no bound on
  that side; with the causal mask the right bound is 0.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, invariants, library routines, brute force and hand-derived
golden values).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "decode_f16", "decode_bf16", "decode",
    "attention_reference", "attention_reference_f64", "attention_rows",
    "softmax_probabilities", "online_softmax_attention", "attention_reference_varlen",
]


# ---------------------------------------------------------------------------
# exact decoding of the 16-bit storage types

def decode_f16(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact; numpy's conversion)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact).

    A bfloat16 value is, by definition, the upper 16 bits of an IEEE binary32
    value whose lower 16 bits are zero.
    """
    b32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b32.view(np.float32).astype(np.float64)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return decode_f16(bits)
    if dtype == "bf16":
        return decode_bf16(bits)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------------------
# the plain definition

def _visible(S: int, rows: np.ndarray, causal: bool, window=(-1, -1)) -> np.ndarray:
    """Boolean mask [len(rows), S]: key j visible to query row i."""
    keys = np.arange(S)[None, :]
    vis = np.ones((len(rows), S), dtype=bool)
    if causal:
        vis &= keys <= rows[:, None]
    left, right = window
    if left >= 0:
        vis &= keys >= rows[:, None] - left
    if right >= 0:
        vis &= keys <= rows[:, None] + right
    return vis


def _rows_one_head(q, k, v, rows, causal, scale, window=(-1, -1)):
    """Definition for query rows ``rows`` of one head.

    q: [S, D], k: [S, D], v: [S, Dv] float64.  Returns (O [n, Dv], LSE [n]).
    """
    S = k.shape[0]
    z = scale * (q[rows] @ k.T)                      # z_ij, fp64
    vis = _visible(S, rows, causal, window)
    z = np.where(vis, z, -np.inf)                   # j outside N_i
    m = z.max(axis=1)                               # M_i
    e = np.exp(z - m[:, None])                      # exp(z_ij - M_i), 0 off N_i
    l = e.sum(axis=1)
    p = e / l[:, None]                              # P_ij
    o = p @ v                                       # O_i
    lse = m + np.log(l)
    return o, lse


def _kv_group(H: int, H_kv: int) -> int:
    """Query heads per K/V head (H_kv must divide H)."""
    if H_kv < 1 or H % H_kv != 0:
        raise ValueError(f"{H_kv} K/V heads do not divide {H} query heads")
    return H // H_kv


def attention_reference_f64(q, k, v, causal: bool, scale: float,
                            row_block: int = 512, window=(-1, -1)):
    """Definition on float64 arrays q [B, S, H, D] and k, v [B, S, H_kv, D].

    Returns (O [B, S, H, D] float64, LSE [B, H, S] float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    group = _kv_group(H, k.shape[2])
    O = np.empty((B, S, H, v.shape[3]), dtype=np.float64)
    LSE = np.empty((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            hk = h // group                              # the K/V head of query head h
            qh, kh, vh = q[b, :, h, :], k[b, :, hk, :], v[b, :, hk, :]
            for r0 in range(0, S, row_block):
                rows = np.arange(r0, min(S, r0 + row_block))
                o, lse = _rows_one_head(qh, kh, vh, rows, causal, scale, window)
                O[b, rows, h, :] = o
                LSE[b, h, rows] = lse
    return O, LSE


def attention_reference(qb, kb, vb, dtype: str, causal: bool, scale: float,
                        window=(-1, -1)):
    """Definition on 16-bit bit arrays [B, S, H, D] (decoded exactly);
    ``window`` = (left, right) keeps keys i - left .. i + right (-1: no bound)."""
    return attention_reference_f64(decode(qb, dtype), decode(kb, dtype),
                                   decode(vb, dtype), causal, scale, window=window)


def attention_rows(qb, kb, vb, dtype: str, causal: bool, scale: float,
                   b: int, h: int, rows, window=(-1, -1)):
    """Definition for a few query rows of one head (full-size sampling).

    Returns (O [len(rows), D], LSE [len(rows)]) in float64.
    """
    rows = np.asarray(rows, dtype=np.int64)
    hk = h // _kv_group(qb.shape[2], kb.shape[2])
    qh = decode(qb[b, :, h, :], dtype)
    kh = decode(kb[b, :, hk, :], dtype)
    vh = decode(vb[b, :, hk, :], dtype)
    return _rows_one_head(qh, kh, vh, rows, causal, scale, window)


def attention_reference_varlen(qb, kb, vb, cu_seqlens, dtype: str, causal: bool, scale: float):
    """Definition on a packed variable-length batch of 16-bit bit arrays:
    each sequence is its own single-batch call of the definition.

    qb [total, H, D], kb / vb [total, H_kv, D], cu_seqlens [B + 1].
    Returns (O [total, H, D], LSE [H, total]) in float64.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total, H, D = qb.shape
    if cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at the token count and not decrease")
    O = np.zeros((total, H, vb.shape[2]), dtype=np.float64)
    LSE = np.zeros((H, total), dtype=np.float64)
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue                                   # an empty sequence has no rows
        o, lse = attention_reference(qb[None, a:e], kb[None, a:e], vb[None, a:e], dtype, causal, scale)
        O[a:e] = o[0]
        LSE[:, a:e] = lse[0]
    return O, LSE


def softmax_probabilities(q, k, causal: bool, scale: float, b: int, h: int):
    """The probability matrix P [S, S] of one head (float64 inputs)."""
    q = np.asarray(q, dtype=np.float64)[b, :, h, :]
    k = np.asarray(k, dtype=np.float64)[b, :, h, :]
    S = k.shape[0]
    rows = np.arange(S)
    z = np.where(_visible(S, rows, causal), scale * (q @ k.T), -np.inf)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# the pages' online recurrence (independent second implementation)

def online_softmax_attention(q, k, v, causal: bool, scale: float,
                             block_n: int, tau: float = 0.0, trace=None,
                             n_tiles=None):
    """Tile-by-tile forward with running (m, l, o~), in fp64.

    q, k, v: float64 arrays [B, S, H, D].  Keys are visited in tiles of
    ``block_n``.  For each tile t with logits s_j (already scaled):

        m_t   = max_j s_j
        m_new = max(m_old, m_t)
        alpha = exp(m_old - m_new)
        p_j   = exp(s_j - m_new)
        l     = alpha * l + sum_j p_j
        o~    = alpha * o~ + sum_j p_j v_j

    and at the end O = o~ / l, LSE = m + ln l.

    ``tau`` > 0 selects the lazy variant: the reference max is only moved
    when the tile max exceeds it by more than ``tau`` (natural-log units);
    otherwise the old reference is kept (alpha = 1) and p_j may exceed 1 by
    at most exp(tau).  Any tau gives the same O and LSE in exact arithmetic.

    ``trace``: optional list; receives (tile_index, m, l, o~) per tile for
    row 0 of head (0, 0).

    ``n_tiles``: by default each row visits only the tiles that hold one of
    its visible keys.  With ``n_tiles`` = T every row visits the first T
    tiles of [0, S) (T >= the tiles holding its last visible key) and the
    keys it may not see are given the logit -inf, so that p_j = 0 for them
    and a tile may be entirely masked.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    Dv = v.shape[3]
    O = np.empty((B, S, H, Dv))
    LSE = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            for i in range(S):
                m = -math.inf
                l = 0.0
                o = np.zeros(Dv)
                last = i if causal else S - 1          # last visible key
                if n_tiles is None:
                    starts = range(0, last + 1, block_n)
                else:
                    assert n_tiles * block_n > last
                    starts = range(0, min(S, n_tiles * block_n), block_n)
                for t, j0 in enumerate(starts):
                    j1 = min(S, j0 + block_n) if n_tiles else min(last + 1, j0 + block_n)
                    s = scale * (k[b, j0:j1, h, :] @ q[b, i, h, :])
                    s = np.where(np.arange(j0, j1) <= last, s, -math.inf)
                    m_t = s.max()
                    m_new = max(m, m_t)
                    if m_new - m > tau or m == -math.inf:
                        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
                        m = m_new
                    else:
                        alpha = 1.0
                    p = np.exp(s - m)
                    l = alpha * l + p.sum()
                    o = alpha * o + p @ v[b, j0:j1, h, :]
                    if trace is not None and b == 0 and h == 0 and i == 0:
                        trace.append((t, m, l, o.copy()))
                O[b, i, h, :] = o / l
                LSE[b, h, i] = m + math.log(l)
    return O, LSE
