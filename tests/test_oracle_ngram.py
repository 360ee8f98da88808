"""Pins for oracle/ngram.py: brute force on tiny histories, invariants, hand-worked drafts."""
import numpy as np
import pytest

from oracle import ngram


def _brute_best(tokens, L, ctx):
    """Rescan the history for one context; best by (count, latest position)."""
    n = len(ctx)
    count, last = {}, {}
    for i in range(n, L):
        if tuple(tokens[i - n:i]) == tuple(ctx):
            c = tokens[i]
            count[c] = count.get(c, 0) + 1
            last[c] = i
    if not count:
        return None
    return max(count, key=lambda c: (count[c], last[c]))


def _brute_draft(tokens, L, max_k):
    seq = list(tokens[:L])
    out = []
    while len(out) < max_k and len(seq) >= 1:
        nxt = _brute_best(tokens, L, seq[-2:]) if len(seq) >= 2 else None
        if nxt is None:
            nxt = _brute_best(tokens, L, seq[-1:])
        if nxt is None:
            break
        out.append(nxt)
        seq.append(nxt)
    return out


@pytest.mark.parametrize("seed", range(40))
def test_matches_brute_force_rescan(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(0, 64))
    V = int(rng.integers(2, 9))
    tokens = list(rng.integers(0, V, size=L))
    tri, bi = ngram.continuation_stats(tokens, L)
    for a in range(V):
        assert (ngram.best_continuation(bi[a]) if a in bi else None) == _brute_best(tokens, L, [a])
        for b in range(V):
            got = ngram.best_continuation(tri[(a, b)]) if (a, b) in tri else None
            assert got == _brute_best(tokens, L, [a, b])
    for max_k in (0, 1, 4, 7):
        assert ngram.draft(tokens, L, max_k) == _brute_draft(tokens, L, max_k)


def test_count_invariants():
    rng = np.random.default_rng(3)
    tokens = list(rng.integers(0, 6, size=500))
    tri, bi = ngram.continuation_stats(tokens, 500)
    assert sum(c for d in bi.values() for c, _ in d.values()) == 499
    assert sum(c for d in tri.values() for c, _ in d.values()) == 498
    # statistics of a prefix grown by appends equal those rebuilt from scratch
    tri2, bi2 = ngram.continuation_stats(tokens, 300)
    assert tri2 != tri
    assert ngram.continuation_stats(tokens[:300], 300) == (tri2, bi2)
    # incremental extension equals the rebuild
    inc = ngram.continuation_stats(tokens, 0)
    prev = 0
    for end in (1, 2, 3, 50, 300, 500):
        ngram.extend_stats(inc, tokens, prev, end)
        prev = end
        assert inc == ngram.continuation_stats(tokens, end)


def test_hand_worked_examples():
    # "a b c a b d a b c": context (a, b) -> c twice, d once => c
    a, b, c, d = 0, 1, 2, 3
    h = [a, b, c, a, b, d, a, b, c, a, b]
    assert ngram.draft(h, len(h), 4) == [c, a, b, c]
    # ties in count go to the most recent occurrence: (x y) -> p at 2, q at 5 => q
    x, y, p, q = 4, 5, 6, 7
    h = [x, y, p, 9, x, y, q, 9, x, y]
    assert ngram.draft(h, len(h), 1) == [q]
    # trigram context unseen -> bigram fallback; bigram unseen -> stop
    h = [1, 2, 3, 8, 2]
    assert ngram.draft(h, len(h), 3) == [3, 8, 2]
    assert ngram.draft([5, 6], 2, 4) == []                 # nothing followed 6
    assert ngram.draft([5], 1, 4) == []
    assert ngram.draft([], 0, 4) == []
    assert ngram.draft([5, 5], 2, 3) == [5, 5, 5]           # self loop


def test_draft_batch_limits_and_padding():
    h = np.array([[0, 1, 0, 1, 0, 1, 0, 0], [3, 3, 3, 3, 0, 0, 0, 0]])
    lens = np.array([7, 4])
    d, n = ngram.draft_batch(h, lens, 4, k_limit=np.array([2, 4]))
    assert list(n) == [2, 4]
    assert list(d[0]) == [1, 0, -1, -1] and list(d[1]) == [3, 3, 3, 3]


def test_fallback_fills_the_positions_after_the_first_miss():
    # With statistics that match the history, a chain either misses at its
    # first step or never misses (every drafted token occurs before the last
    # position, so it has a bigram continuation).  A chain that stops part
    # way needs statistics that lag the history: here they index the prefix
    # [1, 2, 3] while the history has grown to [1, 2, 3, 9, 1].  Context
    # (9, 1): no trigram, bigram 1 -> 2; context (1, 2): trigram -> 3;
    # context (2, 3): no trigram, and 3 was never followed in the indexed
    # prefix -> miss after two drafts.  The fallback proposals then fill
    # positions 2.. of the per-sequence length, i.e. fallback[b, 2:k_b].
    h = np.array([[1, 2, 3, 9, 1, -1, -1, -1]])
    lens = np.array([5])
    stats = [ngram.continuation_stats(h[0], 3)]
    assert ngram.draft(h[0], 5, 4, stats[0]) == [2, 3]
    fb = np.array([[40, 41, 42, 43]])
    cases = {4: [2, 3, 42, 43], 3: [2, 3, 42], 2: [2, 3], 1: [2], 0: []}
    for kb, want in cases.items():
        d, n = ngram.draft_batch(h, lens, 4, k_limit=np.array([kb]), stats=stats, fallback=fb)
        assert int(n[0]) == len(want), (kb, d, n)
        assert list(d[0, :len(want)]) == want and (d[0, len(want):] == -1).all(), (kb, d)
    # a chain that misses at its first step takes the whole cap from the fallback
    d, n = ngram.draft_batch(np.array([[7, 8, -1, -1]]), np.array([2]), 4, k_limit=np.array([3]),
                             fallback=np.array([[50, 51, 52, 53]]))
    assert list(d[0]) == [50, 51, 52, -1] and int(n[0]) == 3
    # without a fallback the chain just stops
    d, n = ngram.draft_batch(h, lens, 4, stats=stats)
    assert list(d[0]) == [2, 3, -1, -1] and int(n[0]) == 2


def test_min_count_needs_repeated_evidence():
    # "repeats n-gram evidence": a context drafts only a continuation seen at least
    # min_count times (worked by hand)
    h = [1, 2, 3, 1, 2, 4, 1, 2]          # (1, 2) -> 3 once, 4 once; 2 -> 3 once, 4 once
    assert ngram.draft(h, len(h), 2) == [4, 1]
    assert ngram.draft(h, len(h), 2, min_count=2) == []
    h = [1, 2, 3, 1, 2, 3, 1, 2]          # (1, 2) -> 3 twice, (2, 3) -> 1 twice, (3, 1) -> 2 twice
    assert ngram.draft(h, len(h), 4, min_count=2) == [3, 1, 2, 3]
    assert ngram.draft(h, len(h), 4, min_count=3) == []
    # the trigram context fails the threshold, the bigram context passes it
    h = [5, 1, 2, 9, 1, 2, 7, 3, 2, 7, 1, 2]  # (1, 2) -> 9 once, 7 once; 2 -> 9, 7, 7: 7 twice
    assert ngram.draft(h, len(h), 1, min_count=2) == [7]
    d, n = ngram.draft_batch(np.array([h]), np.array([len(h)]), 1, min_count=2)
    assert list(d[0]) == [7] and int(n[0]) == 1
