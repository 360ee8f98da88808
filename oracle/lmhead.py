"""The target model's last projection (LM head), fp64 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The verify step takes the target's logits of the K + 1 positions of every
sequence ("SwiftLM: Apple Silicon native MLX Swift LLM inference server",
the paragraph on algorithmic equivalence after Leviathan et al.: the target
model scores the drafts in one forward).  The last operation of that forward
is the LM head, logits = h W^T for the final hidden states h [rows, d] and
the head's weight W [V, d] ("AX Engine: ...", section "Core Technical
Architecture & Methods": the forward's operations run as tensor ops).  The
logits' dtype is bf16, so each dot product is rounded to bf16 (round to
nearest, ties to even) after it is formed.

``lm_head_logits`` forms the dot products in fp64 (a library matmul; exact
for the integer-grid inputs the parity tests use, where every partial sum is
a representable small multiple of a power of two) and rounds them with
``bf16_round``.  Pinned by ``tests/test_oracle_lmhead.py``: hand-worked dot
products, a brute-force triple loop, rounding at hand-worked ties, and the
rounding against torch's own fp32 -> bf16 conversion.
"""
from __future__ import annotations

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (8 significant bits), ties to even.

    Normal range only (|x| in [2^-126, 2^128) or 0); values past the largest
    bf16 go to +-inf.  Returned as fp64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                   # x = m 2^e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0)               # 8 significant bits; rint is half-to-even
    y = np.ldexp(r, e - 8)
    big = np.abs(y) >= 2.0 ** 128
    return np.where(big, np.copysign(np.inf, x), y)


def lm_head_logits(hidden: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """logits[..., v] = bf16_round(sum_i hidden[..., i] weight[v, i]).

    hidden [..., d], weight [V, d] (any float dtype, widened to fp64)."""
    h = np.asarray(hidden, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    return bf16_round(h @ w.T)
