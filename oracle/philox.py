"""Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3" (SC 2011), written from its published definition,
and the dropout keep-mask the kernels draw from it.

TEST INFRASTRUCTURE ONLY (like ``attention_oracle``): the CUDA path has its own
implementation of the same published generator and shares no code with this one.

Philox4x32-R maps a 128-bit counter (x0, x1, x2, x3) and a 64-bit key (k0, k1) to 128
random bits by R rounds of
    (hi0, lo0) = M0 * x0,  (hi1, lo1) = M1 * x2         (32 x 32 -> 64-bit products)
    (x0, x1, x2, x3) <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0)
with the key bumped by the Weyl constants (W0, W1) after each round;
M0 = 0xD2511F53, M1 = 0xCD9E8D57, W0 = 0x9E3779B9, W1 = 0xBB67AE85, R = 10.

Dropout mask (a reading; the pages name dropout for FlashAttention-1 in
"FlashAttention/es", "Variantes y sucesores", but fix no generator): for query head
bh = b * Hq + h, query row i and key j, the counter is (j // 16, i, bh, 0) and the key
is the 64-bit seed (low word first); of the 16 output bytes (word w = byte // 4, bits
8 * (byte % 4) upward) byte j % 16 belongs to key j, and the element is kept iff that
byte is at least floor(256 p), capped at 255: the drop probability is quantised to
1/256. Kept elements are scaled by 1 / (1 - p).

Pinned by tests/test_dropout_oracle.py against the known-answer vectors published with
the generator's reference implementation (Random123), and by mask statistics.
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32(counters, key, rounds: int = 10) -> np.ndarray:
    """counters: [n, 4] (uint32 values), key: (k0, k1). Returns [n, 4] uint32."""
    c = np.asarray(counters, dtype=np.uint64).reshape(-1, 4) & _MASK32
    x0, x1, x2, x3 = (c[:, t].copy() for t in range(4))
    k0, k1 = np.uint64(int(key[0]) & 0xFFFFFFFF), np.uint64(int(key[1]) & 0xFFFFFFFF)
    for _ in range(rounds):
        p0 = np.uint64(M0) * x0
        p1 = np.uint64(M1) * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + np.uint64(W0)) & _MASK32
        k1 = (k1 + np.uint64(W1)) & _MASK32
    return np.stack([x0, x1, x2, x3], axis=1).astype(np.uint32)


def drop_threshold(p: float) -> int:
    """Bytes below this value drop their element: floor(256 p), at most 255."""
    return min(255, int(np.floor(float(p) * 256.0)))


def keep_mask(seed: int, bh: int, rows, cols, p: float) -> np.ndarray:
    """Boolean keep[len(rows), len(cols)] for query head bh."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    blocks = np.unique(cols // 16)
    ii, bb = np.meshgrid(rows, blocks, indexing="ij")                # [R, nb]
    ctr = np.stack([bb.ravel(), ii.ravel(), np.full(ii.size, bh), np.zeros(ii.size)],
                   axis=1).astype(np.uint64)
    words = philox4x32(ctr, key).reshape(len(rows), len(blocks), 4).astype(np.uint32)
    by = np.stack([(words[..., k // 4] >> np.uint32(8 * (k % 4))) & np.uint32(0xFF)
                   for k in range(16)], axis=-1)                      # [R, nb, 16] bytes
    bi = np.searchsorted(blocks, cols // 16)
    vals = by[:, bi, cols % 16]                                       # [R, len(cols)]
    return vals >= drop_threshold(p)
