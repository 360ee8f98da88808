"""Philox4x32-10 and the noise maps of the sampler (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages require a random accept test ("accept when u <= P_target/P_draft",
SwiftLM, paragraph on algorithmic equivalence after Leviathan et al.) and a
resample from the corrected distribution on rejection.  They do not say how
the randomness is produced.  Reading taken here: all randomness is
counter-based, from Philox4x32-10 as published by Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11), keyed by the
64-bit seed, with the counter built from (vocab id, row position, purpose,
step, sequence).  This module is written from that paper's definition and
shares no code with the GPU library, which has its own implementation.

Sampling noise.  The sampler takes argmax_v (log w_v - ln E_v) with E_v
i.i.d. Exp(1), i.e. Gumbel-max with g_v = -ln E_v.  The E_v of the 256
vocab ids of one block (ids 256 b .. 256 b + 255) are drawn through the
Renyi representation of exponential order statistics: the smallest of n
i.i.d. Exp(1) variates is Exp(n); its position is uniform on the n slots
and independent of it; and, the distribution being memoryless, the other
n - 1 exceed it by i.i.d. Exp(1) amounts.  So with one block draw
(M ~ Exp(256), I uniform on 0..255) and one draw F_v ~ Exp(1) per id,

    E_v = M          if v mod 256 == I
    E_v = M + F_v    otherwise,

the E_v are exactly i.i.d. Exp(1), and every score of the block is bounded
by log w_v - ln M.  (Ids beyond the vocabulary fill the last block; their
weight is zero, so they never win.)  An Exp(1) variate is E = -ln u for a
Philox uniform u, taken as -log1p(u - 1) when u > 1/2, where u - 1 is exact.

Counter layout (both sides follow it):

    element draw F_v for vocab id v at row ``pos``:
        counter = (v >> 2, pos | 0 << 16, step mod 2**32, seq), word v & 3
    block draw (M, I) for block b = v >> 8 at row ``pos``:
        counter = (b, pos | 2 << 16, step mod 2**32, seq);
        M = E(word 0) / 256, I = word 1 & 255
    ACCEPT draw for draft i (1-based):
        counter = (0, i | 1 << 16, step mod 2**32, seq), word 0
    key = (seed mod 2**32, seed >> 32)

With u on the 2**-24 grid, g_v lies in about [-2.82, 22.18] (the top end is
-ln of the smallest M); the truncation is a bias of order 2**-24 per draw.

Pinned by: tests/test_oracle_philox.py (against Triton's independent
Philox implementation run on the CPU interpreter, uniformity chi-square,
the exactness of the uniform grid, and the block construction: the law of
the block minimum and of its position, the Exp(1) marginals, and
Gumbel-max against softmax over several blocks).
"""
from __future__ import annotations

import numpy as np

# Multipliers and Weyl key increments of Philox4x32 (Salmon et al. 2011, Sec. 4.1).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

PURPOSE_GUMBEL = 0
PURPOSE_ACCEPT = 1
PURPOSE_BLOCK = 2

NOISE_BLOCK = 256           # vocab ids per block draw (a power of two)
NOISE_BLOCK_SHIFT = 8

_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(m: int, x: np.ndarray):
    """32x32 -> (hi, lo) 32-bit halves of the 64-bit product."""
    p = np.uint64(m) * x
    return p >> np.uint64(32), p & _MASK32


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox4x32 rounds on counter (c0..c3) under key (k0, k1).

    One round (Salmon et al. 2011, Sec. 4.1, the Philox S-box with N = 4):
        (hi0, lo0) = M0 * c0,  (hi1, lo1) = M1 * c2
        c' = (hi1 ^ c1 ^ k0,  lo1,  hi0 ^ c3 ^ k1,  lo0)
    and the key is bumped by the Weyl constants between rounds.
    Inputs broadcast; returns four uint64 arrays holding 32-bit words.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _MASK32 for c in (c0, c1, c2, c3))
    c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for r in range(PHILOX_ROUNDS):
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r + 1 < PHILOX_ROUNDS:
            k0 = np.uint64((int(k0) + PHILOX_W0) & 0xFFFFFFFF)
            k1 = np.uint64((int(k1) + PHILOX_W1) & 0xFFFFFFFF)
    return c0, c1, c2, c3


def seed_key(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniform_from_word(w) -> np.ndarray:
    """u = (2 * (w >> 9) + 1) * 2**-24, the midpoint of one of 2**23 equal cells.

    u lies strictly inside (0, 1), so ln u and ln(-ln u) are finite, and it
    is exact in both fp32 and fp64.
    """
    w = np.asarray(w, dtype=np.uint64)
    m = (w >> np.uint64(9)).astype(np.float64)
    return (2.0 * m + 1.0) * 2.0 ** -24


def exp_from_uniform(u) -> np.ndarray:
    """Exp(1) variate E = -ln u.

    For u > 1/2 the logarithm is taken as log1p(u - 1): u - 1 is exact
    there, which keeps small E (the large Gumbel values that win a
    Gumbel-max) accurate.
    """
    u = np.asarray(u, dtype=np.float64)
    return np.where(u > 0.5, -np.log1p(u - 1.0), -np.log(u))


def gumbel_from_uniform(u) -> np.ndarray:
    """Standard Gumbel variate -ln(-ln u) of one uniform (a single Exp(1) draw)."""
    return -np.log(exp_from_uniform(u))


def _ctr(step, seq, pos, purpose):
    pos = np.asarray(pos, dtype=np.uint64)
    return (pos | np.uint64(purpose << 16), np.uint64(int(step) & 0xFFFFFFFF),
            np.asarray(seq, dtype=np.uint64))


def block_draw(seed: int, seq, step: int, pos, blk):
    """(M, I) of vocab block ``blk`` at row ``pos``: M ~ Exp(256), I uniform on 0..255."""
    k0, k1 = seed_key(seed)
    c1, c2, c3 = _ctr(step, seq, pos, PURPOSE_BLOCK)
    w0, w1, _, _ = philox4x32_10(np.asarray(blk, dtype=np.uint64), c1, c2, c3, k0, k1)
    M = exp_from_uniform(uniform_from_word(w0)) / NOISE_BLOCK
    I = (w1 & np.uint64(NOISE_BLOCK - 1)).astype(np.int64)
    return M, I


def element_exp(seed: int, seq, step: int, pos, v) -> np.ndarray:
    """F_v ~ Exp(1), the per-id draw (before the block minimum is added)."""
    k0, k1 = seed_key(seed)
    v = np.asarray(v, dtype=np.uint64)
    c1, c2, c3 = _ctr(step, seq, pos, PURPOSE_GUMBEL)
    words = philox4x32_10(v >> np.uint64(2), c1, c2, c3, k0, k1)
    lane = (v & np.uint64(3)).astype(np.int64)
    w = np.choose(np.broadcast_to(lane, words[0].shape), words)
    return exp_from_uniform(uniform_from_word(w))


def exp_noise(seed: int, seq, step: int, pos, v) -> np.ndarray:
    """E_v ~ Exp(1) for (seq, step, pos, vocab id v); arguments broadcast."""
    v = np.asarray(v, dtype=np.int64)
    M, I = block_draw(seed, seq, step, pos, v >> NOISE_BLOCK_SHIFT)
    F = element_exp(seed, seq, step, pos, v)
    return np.where((v & (NOISE_BLOCK - 1)) == I, M, M + F)


def gumbel_noise(seed: int, seq, step: int, pos, v) -> np.ndarray:
    """Gumbel noise g_v = -ln E_v for (seq, step, pos, vocab id v); arguments broadcast."""
    return -np.log(exp_noise(seed, seq, step, pos, v))


def exp_row(seed: int, seq, step: int, pos, V: int) -> np.ndarray:
    """E_v for vocab ids 0..V-1 of row ``pos``: shape broadcast(seq, pos) + (V,).

    Same values as ``exp_noise(..., v=arange(V))``; each Philox block is
    evaluated once: four words serve four consecutive ids, one block draw
    serves 256 ids.
    """
    k0, k1 = seed_key(seed)
    seq = np.asarray(seq, dtype=np.uint64)[..., None]
    pos = np.asarray(pos, dtype=np.uint64)[..., None]
    c1, c2, c3 = _ctr(step, seq, pos, PURPOSE_GUMBEL)
    quads = np.arange((V + 3) // 4, dtype=np.uint64)
    words = philox4x32_10(quads, c1, c2, c3, k0, k1)
    w = np.stack(words, axis=-1).reshape(words[0].shape[:-1] + (-1,))[..., :V]
    F = exp_from_uniform(uniform_from_word(w))
    nblk = (V + NOISE_BLOCK - 1) // NOISE_BLOCK
    M, I = block_draw(seed, seq, step, pos, np.arange(nblk, dtype=np.uint64))
    v = np.arange(V)
    Mv = np.repeat(M, NOISE_BLOCK, axis=-1)[..., :V]
    Iv = np.repeat(I, NOISE_BLOCK, axis=-1)[..., :V]
    return np.where((v & (NOISE_BLOCK - 1)) == Iv, Mv, Mv + F)


def gumbel_row(seed: int, seq, step: int, pos, V: int) -> np.ndarray:
    """Gumbel noise -ln E_v for vocab ids 0..V-1 of row ``pos`` (see ``exp_row``)."""
    return -np.log(exp_row(seed, seq, step, pos, V))


def accept_uniform(seed: int, seq, step: int, i) -> np.ndarray:
    """Uniform u_i for the accept test of draft i (1-based) of sequence seq."""
    k0, k1 = seed_key(seed)
    i = np.asarray(i, dtype=np.uint64)
    c1 = i | np.uint64(PURPOSE_ACCEPT << 16)
    w0, _, _, _ = philox4x32_10(np.uint64(0), c1, np.uint64(int(step) & 0xFFFFFFFF),
                                np.asarray(seq, dtype=np.uint64), k0, k1)
    return uniform_from_word(w0)
