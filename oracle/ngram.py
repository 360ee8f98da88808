"""Bigram/trigram continuation statistics and chained drafting (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: AX Engine page, "Core Technical Architecture & Methods": n-gram
speculative decoding builds bigram and trigram tables at runtime from the
tokens seen so far and predicts up to 4 draft tokens per step, with no
second model.  The pages do not fix the lookup rule; the reading used here
(and by the GPU library):

* a continuation of context (t-2, t-1) [trigram] or (t-1) [bigram] is the
  token that followed it somewhere in the history;
* the best continuation of a context has the largest count; equal counts go
  to the continuation whose latest occurrence is the most recent;
* any count >= 1 drafts;
* a draft step looks up the trigram context first, then the bigram context,
  and stops at the first step where neither has a continuation;
* the context of draft step s is the last two tokens of history ++ the drafts
  made so far (drafting is chained), and drafts never change the statistics;
* only tokens that are in the history are indexed (emitted tokens join the
  history through the append step).

This module rebuilds the statistics from the history with plain Python
dictionaries and a linear scan per context, deliberately unlike the GPU's
incremental open-addressed table.

Pinned by: tests/test_oracle_ngram.py (brute-force rescan of tiny histories
for every context, sum-of-counts invariant, chained-draft examples worked by
hand).
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

Stats = Dict[object, Dict[int, List[int]]]


def continuation_stats(tokens: Sequence[int], length: int) -> Tuple[Stats, Stats]:
    """Count, for every context, each continuation and its latest position.

    Returns (tri, bi): tri[(t2, t1)][c] = [count, last_pos] over positions
    i in [2, length) with tokens[i-2], tokens[i-1], tokens[i] = t2, t1, c;
    bi[t1][c] likewise over i in [1, length).
    """
    tri: Stats = {}
    bi: Stats = {}
    for i in range(1, length):
        c = int(tokens[i])
        e = bi.setdefault(int(tokens[i - 1]), {}).setdefault(c, [0, -1])
        e[0] += 1
        e[1] = i
        if i >= 2:
            e = tri.setdefault((int(tokens[i - 2]), int(tokens[i - 1])), {}).setdefault(c, [0, -1])
            e[0] += 1
            e[1] = i
    return tri, bi


def extend_stats(stats: Tuple[Stats, Stats], tokens: Sequence[int], start: int, length: int):
    """Add positions [max(start, 1), length) to (tri, bi); equal to a rebuild."""
    tri, bi = stats
    for i in range(max(start, 1), length):
        c = int(tokens[i])
        e = bi.setdefault(int(tokens[i - 1]), {}).setdefault(c, [0, -1])
        e[0] += 1
        e[1] = i
        if i >= 2:
            e = tri.setdefault((int(tokens[i - 2]), int(tokens[i - 1])), {}).setdefault(c, [0, -1])
            e[0] += 1
            e[1] = i
    return stats


def best_continuation(conts: Dict[int, List[int]], min_count: int = 1):
    """Most frequent continuation, latest occurrence breaking ties; None if there
    is none or if it was seen fewer than ``min_count`` times."""
    best = None
    best_key = None
    for c, (count, last) in conts.items():
        key = (count, last)
        if best_key is None or key > best_key:
            best, best_key = c, key
    if best_key is not None and best_key[0] < min_count:
        return None
    return best


def draft(tokens: Sequence[int], length: int, max_k: int, stats=None, min_count: int = 1) -> List[int]:
    """Chained trigram-then-bigram drafting of up to ``max_k`` tokens.

    ``min_count`` (reading of the AX Engine page's note under the decode table:
    speculation "repeats n-gram evidence"): a context drafts only a
    continuation seen at least that many times; 1 drafts on any evidence."""
    if stats is None:
        stats = continuation_stats(tokens, length)
    tri, bi = stats
    ctx = [int(t) for t in tokens[max(0, length - 2):length]]
    out: List[int] = []
    while len(out) < max_k and len(ctx) >= 1:
        nxt = None
        if len(ctx) >= 2 and (ctx[-2], ctx[-1]) in tri:
            nxt = best_continuation(tri[(ctx[-2], ctx[-1])], min_count)
        if nxt is None and ctx[-1] in bi:
            nxt = best_continuation(bi[ctx[-1]], min_count)
        if nxt is None:
            break
        out.append(nxt)
        ctx = (ctx + [nxt])[-2:]
    return out


def draft_batch(history, lens, max_k: int, k_limit=None, stats=None, fallback=None, min_count: int = 1):
    """Drafts for every sequence: (drafts [B, max_k] padded with -1, counts [B]).

    ``stats`` optionally holds each sequence's statistics of its whole
    history (as kept up to date by ``extend_stats``).  ``fallback`` [B, max_k]
    optionally holds another drafter's proposals: the positions after the
    first miss, up to the per-sequence cap, take them (reading of a
    fixed per-sequence draft length when the tables run dry)."""
    import numpy as np
    B = len(lens)
    drafts = np.full((B, max(max_k, 0)), -1, dtype=np.int64)
    counts = np.zeros(B, dtype=np.int64)
    for b in range(B):
        kb = max_k if k_limit is None else max(0, min(max_k, int(k_limit[b])))
        d = draft(history[b], int(lens[b]), kb, None if stats is None else stats[b], min_count)
        if fallback is not None:
            d = d + [int(t) for t in fallback[b, len(d):kb]]
        drafts[b, :len(d)] = d
        counts[b] = len(d)
    return drafts, counts
