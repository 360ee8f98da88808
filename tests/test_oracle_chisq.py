"""Chi-square pins of the whole oracle verify procedure at V = 32.

The enumeration test checks the rule functions exactly; these tests run the
oracle's full ``spec_verify`` (Philox noise, accept scan, row selection,
Gumbel-max residual / bonus) over 10**6 seeded steps and compare the joint
law of (accept length a, sampled token y) with its closed form:

    point mass:  P(a, y) = prod_{j<a} p_j(d_{j+1}) * (p_a(y) [y != d_{a+1}]  if a < k
                                                     p_k(y)                  if a = k)
    dense q:     P(a, y) = prod_{j<a} alpha_j * (max(0, p_a(y) - q_a(y))     if a < k
                                                 p_k(y)                      if a = k)
                 with alpha_j = sum_v min(p_j(v), q_j(v))

(Leviathan et al.; SwiftLM page, paragraph on algorithmic equivalence).
Steps are independent draws because the noise counter includes the step
and the sequence id; the test varies both.
"""
import numpy as np
import pytest
from scipy import stats

from oracle import philox
from oracle import verify as ov
from oracle.verify import VerifyParams

V, K = 32, 4
N_STEPS = 10 ** 6
CHUNK = 100_000


def _rows(seed, T):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0.0, 3.0, size=(K + 1, V)) * T
    return logits


def _chisq(observed, expected, min_expected=5.0):
    small = expected < min_expected
    obs = np.append(observed[~small], observed[small].sum())
    exp = np.append(expected[~small], expected[small].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp * obs.sum() / exp.sum()).pvalue


def _run(logits_rows, drafts_fn, q_rows, params, n_steps):
    counts = np.zeros((K + 1, V))
    for c in range(n_steps // CHUNK):
        B = CHUNK
        logits = np.broadcast_to(logits_rows, (B, K + 1, V))
        drafts = drafts_fn(c, B)
        dp = None if q_rows is None else np.broadcast_to(q_rows, (B, K, V))
        p = VerifyParams(**{**params.__dict__, "step": params.step + c})
        res = ov.spec_verify(logits, drafts, dp, np.full(B, K), np.zeros((B, 1), int),
                             np.zeros(B, int), p, np.zeros(B), np.ones(B),
                             seq_ids=np.arange(B) + 7 * c)
        a = res["accept_len"]
        y = res["out_tokens"][np.arange(B), a]
        np.add.at(counts, (a, y), 1)
    return counts


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_point_mass_joint_law(T):
    logits = _rows(31, T)
    p = np.exp(ov.log_softmax(logits / float(np.float32(T))))
    # drafts with a spread of acceptance probabilities so every a is visited
    d = np.array([int(np.argsort(p[j])[-1 - (j % 2)]) for j in range(K)])
    expected = np.zeros((K + 1, V))
    reach = 1.0
    for a in range(K + 1):
        if a < K:
            row = p[a].copy()
            row[d[a]] = 0.0
            expected[a] = reach * row
            reach *= p[a, d[a]]
        else:
            expected[a] = reach * p[K]
    assert abs(expected.sum() - 1) < 1e-12
    params = VerifyParams(temperature=T, gate_enabled=False, seed=2024, step=0)
    counts = _run(logits, lambda c, B: np.broadcast_to(d, (B, K)), None, params, N_STEPS)
    pv = _chisq(counts.ravel(), expected.ravel() * N_STEPS)
    assert pv > 1e-3, pv


def test_dense_joint_law():
    T = 0.6
    logits = _rows(57, T)
    rng = np.random.default_rng(58)
    q_logits = logits[:K] + rng.normal(0, 0.5, size=(K, V))
    q = np.exp(q_logits / T - (q_logits / T).max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    p = np.exp(ov.log_softmax(logits / float(np.float32(T))))
    # q is stored as fp32 by the library; use the same values here
    q = q.astype(np.float32).astype(np.float64)
    alpha = np.minimum(p[:K], q).sum(-1)
    expected = np.zeros((K + 1, V))
    reach = 1.0
    for a in range(K + 1):
        expected[a] = reach * (np.maximum(0.0, p[a] - q[a]) if a < K else p[K])
        if a < K:
            reach *= alpha[a]
    assert abs(expected.sum() - 1) < 1e-6
    draw_rng = np.random.default_rng(99)
    cdf = np.cumsum(q, axis=-1)

    def drafts_fn(c, B):
        u = draw_rng.random((B, K))
        return np.stack([np.minimum(np.searchsorted(cdf[j], u[:, j] * cdf[j, -1]), V - 1)
                         for j in range(K)], axis=1)

    params = VerifyParams(temperature=T, gate_enabled=False, seed=77, step=5)
    counts = _run(logits, drafts_fn, q, params, N_STEPS)
    pv = _chisq(counts.ravel(), expected.ravel() * N_STEPS)
    assert pv > 1e-3, pv


def test_gumbel_max_matches_softmax():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 2, size=V)
    logp = ov.log_softmax(x)
    n = 10 ** 6
    seq = np.arange(n)
    g = philox.gumbel_noise(5, seq[:, None], 3, 1, np.arange(V)[None, :])
    y, _ = ov.gumbel_argmax(np.broadcast_to(logp, (n, V)), g)
    counts = np.bincount(y, minlength=V)
    assert _chisq(counts, np.exp(logp) * n) > 1e-3


def test_sample_and_match_has_the_same_law():
    """Cross-check (point mass): accepting d iff d = argmax(x/T + g) is another
    procedure with the same law; its (a, y) histogram must agree with the
    oracle's u-test procedure (two-sample chi-square)."""
    T = 1.0
    logits = _rows(13, T)
    lp = ov.log_softmax(logits / T)
    d = np.array([int(np.argmax(lp[j])) for j in range(K)])
    n = 400_000
    params = VerifyParams(temperature=T, gate_enabled=False, seed=31, step=0)
    ours = _run(logits, lambda c, B: np.broadcast_to(d, (B, K)), None, params, n)
    # sample-and-match: row j draws y_j by Gumbel-max; accept while y_j == d_{j+1}
    seq = np.arange(n) + 10 ** 7
    alt = np.zeros((K + 1, V))
    alive = np.ones(n, dtype=bool)
    for j in range(K + 1):
        g = philox.gumbel_noise(999, seq[:, None], 1, j, np.arange(V)[None, :])
        y, _ = ov.gumbel_argmax(np.broadcast_to(lp[j], (n, V)), g)
        stop = alive & ((y != d[j]) if j < K else True)
        np.add.at(alt, (np.full(stop.sum(), j), y[stop]), 1)
        alive &= ~stop
    table = np.stack([ours.ravel(), alt.ravel()])
    table = table[:, table.sum(0) > 0]
    small = table.sum(0) < 10
    table = np.concatenate([table[:, ~small], table[:, small].sum(1, keepdims=True)], axis=1)
    assert stats.chi2_contingency(table)[1] > 1e-3
