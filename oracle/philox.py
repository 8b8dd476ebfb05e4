"""Philox4x32-10 counter-based generator, written from its published definition.

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11, section on the Philox S-box: each round
multiplies two of the four 32-bit counter words by fixed constants, swaps the
words and xors the high product halves with the other words and the key; the
two key words are bumped by Weyl constants (golden ratio, sqrt(3)-1) between
rounds; Philox4x32-10 runs ten rounds.

The EAGLE pages do not fix a random-number generator. The speculative sampling
rule needs uniform draws (accept/reject tests, the bonus token, planted-mode
draws); both sides of the parity tests implement this one generator so that
draws agree bit for bit. The keying scheme (which counter words carry which
indices) is this build's own convention and is repeated on the CUDA side.

Test infrastructure: only tests, the smoke check and the bench's CPU baseline
use this package.
"""
from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint64(0x9E3779B9)
W1 = np.uint64(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)

# stream ids of the draws this method makes (low byte of counter word 3)
STREAM_PLANT = 2
STREAM_ACCEPT = 3
STREAM_GUMBEL = 4
STREAM_PLAIN = 5
PREFILL_CYCLE = 0xFFFFFFFF   # cycle index used for the first token drawn at prefill


def philox4x32_10(ctr, key):
    """ctr: uint array [..., 4], key: uint array [..., 2] -> uint32 array [..., 4]."""
    c = [np.asarray(ctr[..., i], dtype=np.uint64) & MASK32 for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64) & MASK32
    k1 = np.asarray(key[..., 1], dtype=np.uint64) & MASK32
    for r in range(10):
        if r > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c[0]
        p1 = M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack(c, axis=-1).astype(np.uint32)


def key_of(seed: int):
    """The Philox4x32 key (two 32-bit words, low word first) of a 64-bit seed."""
    return np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)


def to_uniform(x):
    """23-bit uniform strictly inside (0, 1): ((x >> 9) + 0.5) * 2^-23, exactly
    representable in fp32 (the largest value is 1 - 2^-24)."""
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * (2.0 ** -23)


def draw_uniform(seed: int, stream: int, seq: int, cycle: int, a: int, b: int) -> float:
    """One uniform keyed by (seed; counter = (a, b, cycle, seq << 8 | stream)), word 0."""
    ctr = np.array([a, b, cycle & 0xFFFFFFFF, (seq << 8) | stream], dtype=np.uint64)
    return float(to_uniform(philox4x32_10(ctr, key_of(seed))[0]))


def gumbel_row(seed: int, stream: int, seq: int, cycle: int, row: int, vocab: int) -> np.ndarray:
    """Gumbel(0,1) noise for every vocabulary id v of one row: uniform from
    counter (v >> 2, row, cycle, seq << 8 | stream), word v & 3; g = -log(-log(u))."""
    v = np.arange(vocab, dtype=np.uint64)
    n = (vocab + 3) // 4
    ctr = np.zeros((n, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(n, dtype=np.uint64)
    ctr[:, 1] = row
    ctr[:, 2] = cycle & 0xFFFFFFFF
    ctr[:, 3] = (seq << 8) | stream
    out = philox4x32_10(ctr, np.broadcast_to(key_of(seed), (n, 2)))
    u = to_uniform(out.reshape(-1)[:vocab])
    del v
    return -np.log(-np.log(u))
