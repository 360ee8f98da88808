"""Exact enumeration pin (V = 8, K <= 3) of the oracle's accept and residual rules.

Leviathan/Chen's claim (SwiftLM page, paragraph on algorithmic equivalence):
speculative sampling emits tokens distributed exactly as the target.  Here
the law of one verify step is computed exactly from the oracle's own rule
functions -- ``accept_draft`` counted over the 2**23-point grid of u and
``residual_weights`` normalised -- by walking every draft tuple.  Completing
each emitted prefix with target samples up to K + 1 tokens must give the
target's joint law prod_i p(t_i | t_<i), up to the grid error (about 2**-23
per accept factor).  The target conditionals are computed here with plain
numpy, not with the oracle.
"""
import itertools

import numpy as np
import pytest

from oracle import verify as ov

V = 8
GRID = 2 ** 23


def _u(m):
    return (2.0 * m + 1.0) * 2.0 ** -24


def accept_prob(p_d, q_d):
    """P(u * q <= p) over the u grid, by bisection on the oracle's rule (monotone in u)."""
    coarse = np.array([bool(ov.accept_draft(_u(m), p_d, q_d)) for m in range(0, GRID, GRID // 64)])
    assert (np.diff(coarse.astype(int)) <= 0).all(), "accept rule is not monotone in u"
    lo, hi = 0, GRID                     # invariant: rule holds below lo, fails at hi (or hi == GRID)
    if not ov.accept_draft(_u(0), p_d, q_d):
        return 0.0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ov.accept_draft(_u(mid), p_d, q_d):
            lo = mid
        else:
            hi = mid
    return hi / GRID


class Model:
    """Seeded target (and draft-model) conditionals over V = 8 ids."""

    def __init__(self, seed, T):
        self.seed, self.T = seed, T
        self.cache = {}

    def _logits(self, prefix, which):
        key = (which,) + tuple(prefix)
        if key not in self.cache:
            rng = np.random.default_rng([self.seed, which] + [t + 1 for t in prefix])
            self.cache[key] = rng.normal(0.0, 1.5, size=V)
        return self.cache[key]

    def target(self, prefix):
        """Target conditional p(. | prefix), plain numpy softmax."""
        key = ("p",) + tuple(prefix)
        if key not in self.cache:
            y = self._logits(prefix, 0) / self.T
            e = np.exp(y - y.max())
            self.cache[key] = e / e.sum()
        return self.cache[key]

    def target_via_oracle(self, prefix):
        """The same distribution as the oracle's verify computes it."""
        return np.exp(ov.log_softmax(self._logits(prefix, 0) / self.T))

    def draft(self, prefix):
        """Draft-model conditional q(. | prefix): target logits plus noise."""
        y = (self._logits(prefix, 0) + 0.7 * self._logits(prefix, 1)) / self.T
        e = np.exp(y - y.max())
        return e / e.sum()


def step_law(model, k, drafts_and_weights, dense):
    """Exact law of (emitted prefix) for one verify step, from the oracle's rules."""
    law = {}
    for drafts, w in drafts_and_weights:
        reach = w
        for a in range(k + 1):
            prefix = tuple(drafts[:a])
            p_a = model.target_via_oracle(prefix)
            if a == k:
                for y in range(V):                      # all accepted: bonus from p_k
                    e = prefix + (y,)
                    law[e] = law.get(e, 0.0) + reach * p_a[y]
                break
            d = drafts[a]
            q_row = model.draft(prefix) if dense else np.eye(V)[d]
            A = accept_prob(p_a[d], q_row[d])
            r = ov.residual_weights(p_a, q_row)
            if r.sum() == 0:
                r = p_a
            r = r / r.sum()
            for y in range(V):                          # rejected: residual sample
                e = prefix + (y,)
                law[e] = law.get(e, 0.0) + reach * (1.0 - A) * r[y]
            reach *= A
    return law


def completed_joint(model, k, law):
    """Extend each emitted prefix with target samples to length k + 1."""
    joint = np.zeros((V,) * (k + 1))
    for e, pe in law.items():
        if pe == 0.0:
            continue
        rest = k + 1 - len(e)
        for tail in itertools.product(range(V), repeat=rest):
            t = e + tail
            pr = pe
            for i in range(len(e), k + 1):
                pr *= model.target(t[:i])[t[i]]
            joint[t] += pr
    return joint


def target_joint(model, k):
    joint = np.zeros((V,) * (k + 1))
    for t in itertools.product(range(V), repeat=k + 1):
        pr = 1.0
        for i in range(k + 1):
            pr *= model.target(t[:i])[t[i]]
        joint[t] = pr
    return joint


def _point_mass_tuples(k, n, seed):
    allt = list(itertools.product(range(V), repeat=k))
    if len(allt) <= n:
        return allt
    rng = np.random.default_rng(seed)
    return [allt[i] for i in rng.choice(len(allt), size=n, replace=False)]


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("T", [1.0, 0.6])
def test_point_mass_drafts_emit_the_target_law(k, T):
    model = Model(seed=100 + k, T=T)
    ref = target_joint(model, k)
    for drafts in _point_mass_tuples(k, 24, seed=k):
        joint = completed_joint(model, k, step_law(model, k, [(tuple(drafts), 1.0)], dense=False))
        assert abs(joint.sum() - 1.0) < 1e-9
        np.testing.assert_allclose(joint, ref, rtol=0, atol=k * 2.0 ** -22)


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("T", [1.0, 0.6])
def test_dense_drafts_emit_the_target_law(k, T):
    model = Model(seed=200 + k, T=T)
    tuples = []
    for drafts in itertools.product(range(V), repeat=k):
        w = 1.0
        for i in range(k):
            w *= model.draft(drafts[:i])[drafts[i]]
        tuples.append((drafts, w))
    joint = completed_joint(model, k, step_law(model, k, tuples, dense=True))
    ref = target_joint(model, k)
    assert abs(joint.sum() - 1.0) < 1e-9
    np.testing.assert_allclose(joint, ref, rtol=0, atol=k * 2.0 ** -22)


def test_enumeration_detects_a_planted_mistake(monkeypatch):
    """The pin has teeth: a wrong accept rule planted in the oracle fails it."""
    model = Model(seed=7, T=1.0)
    k = 1
    ref = target_joint(model, k)
    monkeypatch.setattr(ov, "accept_draft", lambda u, p, q: np.asarray(u) * np.asarray(q) <= 0.5 * np.asarray(p))
    bad = completed_joint(model, k, step_law(model, k, [((3,), 1.0)], dense=False))
    assert np.abs(bad - ref).max() > 1e-3
    monkeypatch.undo()
    monkeypatch.setattr(ov, "residual_weights", lambda p, q: p)          # residual without max(0, p - q)
    tuples = [((d,), model.draft(())[d]) for d in range(V)]
    bad = completed_joint(model, k, step_law(model, k, tuples, dense=True))
    assert np.abs(bad - ref).max() > 1e-3
