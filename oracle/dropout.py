"""Attention dropout in the fp64 oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; it shares no code with the CUDA path.

Reading (the pages list dropout among the needs of a production FA2 forward,
page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与 TiledMMA",
section 哪些结论可以迁移，哪些只是本例特例, without a formula): every
probability P_ij is kept with probability 1 - p and scaled by 1 / (1 - p)
before it multiplies V, so O_i = sum_j P_ij keep_ij V_j / (1 - p); the row
sums, the max and the LSE are those of the undropped softmax.

The random numbers come from the counter-based generator Philox4x32-10
(J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random numbers: as easy
as 1, 2, 3", SC 2011), written here from its definition: a 128-bit counter
(c0, c1, c2, c3) and a 64-bit key (k0, k1), ten rounds of
    (hi0, lo0) = M0 * c0,  (hi1, lo1) = M1 * c2            (32 x 32 -> 64 bits)
    c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)
with M0 = 0xD2511F53, M1 = 0xCD9E8D57, and the key bumped by
(0x9E3779B9, 0xBB67AE85) before every round but the first.

Each 32-bit output word holds two 16-bit draws (low half first), so one
block serves eight keys: element (b, h, i, j) (query row i, key j) takes
draw j mod 8 -- half j mod 2 of word (j mod 8) div 2 -- of the block with
counter (j div 8, i, h, b) and key (seed mod 2^32, seed div 2^32); it is
kept iff that draw >= floor(p * 2^16) -- an integer decision, the same on
any machine.  (p is thereby taken to a multiple of 2^-16: the keep
probability is 1 - floor(p * 2^16) / 2^16, within 2^-16 of 1 - p; the kept
values are scaled by 1 / (1 - p) as asked.)  Parity status: pinned by tests/test_oracle.py (the generator's
published known-answer vectors, p = 0, the kept fraction, unbiasedness, and
the mask read back through a one-hot V).
"""
from __future__ import annotations

import math

import numpy as np

from .attention import _kv_group, _visible, decode

__all__ = ["philox4x32_10", "dropout_threshold", "dropout_draws", "dropout_keep",
           "attention_reference_dropout"]

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint64(0x9E3779B9), np.uint64(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on arrays of 32-bit counter words (any integer dtype);
    returns the four 32-bit output words as uint64 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in (c0, c1, c2, c3)]
    k0, k1 = np.uint64(k0) & _MASK, np.uint64(k1) & _MASK
    for r in range(10):
        if r > 0:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        c = [(p1 >> _S32) ^ c[1] ^ k0, p1 & _MASK, (p0 >> _S32) ^ c[3] ^ k1, p0 & _MASK]
    return c


def dropout_threshold(p_drop: float) -> int:
    """floor(p * 2^16), the smallest kept 16-bit draw."""
    if not (0.0 <= p_drop < 1.0):
        raise ValueError("p_drop must be in [0, 1)")
    return min(int(math.floor(p_drop * 65536.0)), 65535)


def dropout_draws(b: int, h: int, rows, ng: int, seed: int) -> np.ndarray:
    """The 16-bit draws of head (b, h) for the given query rows and keys
    0 .. 8 * ng - 1, shape [len(rows), 8 * ng]."""
    rows = np.asarray(rows, dtype=np.uint64)
    n = len(rows)
    k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
    g = np.broadcast_to(np.arange(ng, dtype=np.uint64)[None, :], (n, ng))
    i = np.broadcast_to(rows[:, None], (n, ng))
    words = philox4x32_10(g, i, np.full((n, ng), h, dtype=np.uint64),
                          np.full((n, ng), b, dtype=np.uint64), k0, k1)
    w = np.stack(words, axis=-1)                                  # [n, ng, 4]
    halves = np.stack([w & 0xFFFF, w >> np.uint64(16)], axis=-1)  # [n, ng, 4, 2]
    return halves.reshape(n, 8 * ng)      # key 8 g + 2 word + half


def dropout_keep(B: int, H: int, S: int, p_drop: float, seed: int) -> np.ndarray:
    """keep[b, h, i, j] for query rows i and keys j of an S x S score matrix."""
    t = np.uint64(dropout_threshold(p_drop))
    ng = (S + 7) // 8
    keep = np.empty((B, H, S, S), dtype=bool)
    for b in range(B):
        for h in range(H):
            keep[b, h] = dropout_draws(b, h, np.arange(S), ng, seed)[:, :S] >= t
    return keep


def attention_reference_dropout(qb, kb, vb, dtype: str, causal: bool, scale: float,
                                p_drop: float, seed: int):
    """Definition with dropout on 16-bit bit arrays q [B, S, H, D] and k, v
    [B, S, H_kv, D].  Returns (O [B, S, H, D], LSE [B, H, S]) in float64."""
    q, k, v = decode(qb, dtype), decode(kb, dtype), decode(vb, dtype)
    B, S, H, D = q.shape
    group = _kv_group(H, k.shape[2])
    keep = dropout_keep(B, H, S, p_drop, seed)
    rows = np.arange(S)
    vis = _visible(S, rows, causal)
    O = np.empty((B, S, H, v.shape[3]), dtype=np.float64)
    LSE = np.empty((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            hk = h // group
            z = np.where(vis, scale * (q[b, :, h, :] @ k[b, :, hk, :].T), -np.inf)
            m = z.max(axis=1)
            e = np.exp(z - m[:, None])
            l = e.sum(axis=1)
            p = e / l[:, None]
            O[b, :, h, :] = (p * keep[b, h]) @ v[b, :, hk, :] / (1.0 - p_drop)
            LSE[b, h, :] = m + np.log(l)
    return O, LSE
