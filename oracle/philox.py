"""Philox4x32-10 and the dropout keep-mask built from it, in NumPy.

TEST INFRASTRUCTURE (same import rule as ``oracle/attention.py``).

The generator is the counter-based Philox4x32 of Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011), with ten
rounds: a 128-bit counter (four 32-bit words) and a 64-bit key (two words);
each round multiplies counter words 0 and 2 by the round multipliers, keeps
both halves of the 64-bit products, and mixes in the other two words and the
round key; the key is bumped by the Weyl constants between rounds.

Dropout mask (the reading for this library; the pages only name dropout as
an argument of the SDPA call): score (i, j) of unit u = b * H + h is kept iff
byte (j mod 16) of Philox4x32-10(counter = (j // 16, i, u, 0), key = (seed
mod 2^32, seed // 2^32)) is at least t = round(p * 256); bytes are taken
little-endian within each 32-bit output word. Kept probabilities are scaled
by 256 / (256 - t), the inverse of the realised keep rate.
"""
from __future__ import annotations

import numpy as np

__all__ = ["philox4x32_10", "dropout_threshold", "dropout_keep"]

_M0, _M1 = 0xD2511F53, 0xCD9E8D57          # round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85          # key increments (Weyl sequence)
_MASK = np.uint64(0xFFFFFFFF)


def _mulhilo(a: int, x: np.ndarray):
    prod = np.uint64(a) * x.astype(np.uint64)
    return (prod >> np.uint64(32)).astype(np.uint32), (prod & _MASK).astype(np.uint32)


def philox4x32_10(counter, key):
    """counter: uint32 array [..., 4]; key: uint32 array [..., 2] (broadcast).
    Returns the four 32-bit output words [..., 4]."""
    c = np.array(counter, dtype=np.uint32)
    k = np.broadcast_to(np.array(key, dtype=np.uint32), c.shape[:-1] + (2,)).copy()
    c0, c1, c2, c3 = (c[..., n].copy() for n in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0.astype(np.uint64) + _W0).astype(np.uint32)
            k1 = (k1.astype(np.uint64) + _W1).astype(np.uint32)
        hi0, lo0 = _mulhilo(_M0, c0)
        hi1, lo1 = _mulhilo(_M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1)


def dropout_threshold(p: float) -> int:
    """t = round(p * 256): bytes below t drop their score. 0 <= p < 1."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(int(round(p * 256.0)), 255)


def dropout_keep(seed: int, unit: int, lq: int, lk: int, p: float) -> np.ndarray:
    """Boolean keep-mask [lq, lk] of one (batch, head) unit."""
    t = dropout_threshold(p)
    groups = -(-lk // 16)
    i = np.arange(lq, dtype=np.uint32)[:, None]
    g = np.arange(groups, dtype=np.uint32)[None, :]
    ctr = np.stack(np.broadcast_arrays(g, i, np.uint32(unit), np.uint32(0)), axis=-1).astype(np.uint32)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint32)
    words = philox4x32_10(ctr, key)                      # [lq, groups, 4]
    by = words.astype("<u4").view(np.uint8).reshape(lq, groups * 16)[:, :lk]
    return by >= t
