"""Philox4x32-10 counter-based generator, vectorised over numpy arrays.

Written from the published definition in Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 3.3 (the
Philox S-box: two 32x32->64 multiplies per round, the high halves xored with
the other two counter words and the round key, a Weyl-sequence key schedule).

Everything the verification method draws at random (the accept-test uniforms
and the final-sample uniform) is generated here on the host and handed to both
the oracle and the GPU library as plain input arrays, so neither side carries
a generator of its own.
"""
from __future__ import annotations

import numpy as np

# Round multipliers and key-schedule (Weyl) increments of Philox4x32.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# Stream identifiers folded into the high key word so that independent uses
# of one seed never share counters.
STREAM_UNIFORMS = 0x5EED0001
STREAM_DRAFT = 0x5EED0002
STREAM_LOGITS = 0x5EED0003


def philox4x32_10(counter: np.ndarray, key) -> np.ndarray:
    """Apply ten Philox4x32 rounds to each 128-bit counter.

    counter: uint32 array of shape (N, 4).  key: two uint32 words (k0, k1).
    Returns a uint32 array of shape (N, 4).
    """
    ctr = np.asarray(counter, dtype=np.uint32)
    if ctr.ndim != 2 or ctr.shape[1] != 4:
        raise ValueError("counter must have shape (N, 4)")
    c0, c1, c2, c3 = (ctr[:, j].astype(np.uint64) for j in range(4))
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        prod0 = m0 * c0          # 32x32 -> 64 bits, exact in uint64
        prod1 = m1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & _MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def u32_to_unit_float(words: np.ndarray) -> np.ndarray:
    """Map uint32 words to float32 uniforms k * 2^-24 in [0, 1 - 2^-24].

    The top 24 bits are kept, so every value is exactly representable in
    float32 and in float64 alike.
    """
    w = np.asarray(words, dtype=np.uint32)
    return ((w >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def uniform_grid(seed: int, stream: int, rows: int, cols: int) -> np.ndarray:
    """float32 [rows, cols] uniforms; entry (r, c) uses counter (r, c, 0, 0)."""
    r = np.repeat(np.arange(rows, dtype=np.uint64), cols)
    c = np.tile(np.arange(cols, dtype=np.uint64), rows)
    ctr = np.zeros((rows * cols, 4), dtype=np.uint32)
    ctr[:, 0] = (r & _MASK32).astype(np.uint32)
    ctr[:, 1] = (c & _MASK32).astype(np.uint32)
    ctr[:, 2] = (r >> np.uint64(32)).astype(np.uint32)
    key = (int(seed) & 0xFFFFFFFF, (int(stream) ^ (int(seed) >> 32)) & 0xFFFFFFFF)
    out = philox4x32_10(ctr, key)[:, 0]
    return u32_to_unit_float(out).reshape(rows, cols)
