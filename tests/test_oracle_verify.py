"""Pins for oracle/verify.py: closed forms, greedy matching and invariants."""
import json
import os

import numpy as np
import pytest

from oracle import verify as ov
from oracle.verify import VerifyParams

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _argmax_matching(rows, drafts, k):
    """Independent greedy reference: accept while d_{i} is the row argmax."""
    a = 0
    while a < k and drafts[a] == int(np.argmax(rows[a])):
        a += 1
    return a, int(np.argmax(rows[a]))


@pytest.mark.parametrize("seed", range(6))
def test_greedy_equals_argmax_matching(seed):
    rng = np.random.default_rng(seed)
    B, K, V = 64, 4, 50
    # coarse values make exact ties common (as with bf16 logits)
    logits = np.round(rng.normal(0, 2, size=(B, K + 1, V)) * 2) / 2
    am = np.argmax(logits, axis=-1)
    drafts = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K)))
    k = rng.integers(0, K + 1, size=B)
    hist = np.zeros((B, 4), dtype=np.int64)
    p = VerifyParams(temperature=0.0, gate_enabled=False, seed=seed, step=3)
    res = ov.spec_verify(logits, drafts, None, k, hist, np.zeros(B, int), p,
                         np.full(B, 100), np.ones(B, np.float32))
    for b in range(B):
        a, y = _argmax_matching(logits[b], drafts[b], k[b])
        assert res["accept_len"][b] == a
        assert res["out_tokens"][b, a] == y
        assert list(res["out_tokens"][b, :a]) == list(drafts[b, :a])
        assert (res["out_tokens"][b, a + 1:] == -1).all()
        assert res["kv_len"][b] == 100 - k[b] + a


def test_greedy_dense_q_is_argmax_matching_too():
    rng = np.random.default_rng(5)
    B, K, V = 32, 3, 20
    logits = rng.normal(0, 3, size=(B, K + 1, V))
    q = rng.dirichlet(np.ones(V), size=(B, K))
    am = np.argmax(logits, axis=-1)
    drafts = np.where(rng.random((B, K)) < 0.6, am[:, :K], rng.integers(0, V, (B, K)))
    p = VerifyParams(temperature=0.0, gate_enabled=False)
    res = ov.spec_verify(logits, drafts, q, np.full(B, K), np.zeros((B, 1), int), np.zeros(B, int),
                         p, np.zeros(B), np.ones(B))
    for b in range(B):
        a, y = _argmax_matching(logits[b], drafts[b], K)
        assert res["accept_len"][b] == a and res["out_tokens"][b, a] == y


def test_softcap_closed_forms():
    c = 30.0
    x = np.array([0.0, c * np.arctanh(0.5), -c * np.arctanh(0.25), 1e6, -1e6])
    got = ov.softcap(x, c)
    np.testing.assert_allclose(got, [0.0, 15.0, -7.5, 30.0, -30.0], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(ov.softcap(x, 0.0), x)      # off
    np.testing.assert_array_equal(ov.softcap(x, -1.0), x)


def test_repetition_penalty_closed_forms():
    x = np.array([2.2, -1.0, 3.0, 0.0, 5.0])
    got = ov.repetition_penalty(x, np.array([0, 1, 3]), 1.1)
    np.testing.assert_allclose(got, [2.0, -1.1, 3.0, 0.0, 5.0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(ov.repetition_penalty(x, np.array([0, 1]), 1.0), x)
    # each distinct id once: a window holding an id twice penalises it once
    ids = ov.penalty_ids(np.array([4, 4, 0, 9, 9]), 5, np.array([0, 4]), 2, 4)
    assert list(ids) == [0, 4, 9]
    once = ov.repetition_penalty(x, ids[ids < 5], 1.1)
    assert once[4] == 5.0 / 1.1


def test_penalty_window_covers_drafts():
    hist = np.array([1, 2, 3, 4, 5, 6])
    d = np.array([7, 8, 9])
    assert list(ov.penalty_ids(hist, 6, d, 0, 3)) == [4, 5, 6]
    assert list(ov.penalty_ids(hist, 6, d, 2, 3)) == [6, 7, 8]
    assert list(ov.penalty_ids(hist, 2, d, 1, 8)) == [1, 2, 7]
    assert ov.penalty_ids(hist, 6, d, 2, 0).size == 0


def test_transform_order_softcap_then_penalty_then_temperature():
    logits = np.array([[[40.0, -40.0, 1.0]]])
    p = VerifyParams(temperature=0.5, softcap=30.0, rep_penalty=1.25, rep_window=2)
    z = ov.transform_rows(logits, p, np.array([[0, 1]]), np.array([2]), np.zeros((1, 0), int))
    sc = 30.0 * np.tanh(np.array([40.0, -40.0]) / 30.0)
    np.testing.assert_allclose(z[0, 0, :2], [sc[0] / 1.25, sc[1] * 1.25], rtol=1e-15)
    assert z[0, 0, 2] == 30.0 * np.tanh(1.0 / 30.0)


def test_log_softmax_matches_definition():
    y = np.array([[1.0, 2.0, 3.0], [1000.0, 1000.0, -1000.0]])
    lp = ov.log_softmax(y)
    np.testing.assert_allclose(np.exp(lp[0]), np.exp(y[0]) / np.exp(y[0]).sum(), rtol=1e-15)
    np.testing.assert_allclose(lp[1, :2], [-np.log(2)] * 2, rtol=0, atol=2e-13)  # y - lse at |y| = 1000


def test_accept_rule_and_residual():
    assert ov.accept_draft(0.3, 0.3, 1.0) and not ov.accept_draft(0.30001, 0.3, 1.0)
    assert ov.accept_draft(0.99, 0.0, 0.0)                   # q(d) = 0 accepts
    assert ov.accept_draft(0.5, 0.2, 0.4) and not ov.accept_draft(0.6, 0.2, 0.4)
    np.testing.assert_array_equal(ov.residual_weights(np.array([0.5, 0.3, 0.2]), np.array([0.2, 0.5, 0.3])),
                                  [0.3, 0.0, 0.0])


@pytest.mark.parametrize("rho", [0.0, 0.25, 1.0])
def test_ema_closed_form(rho):
    """ema_n = rho + (ema_0 - rho) (1 - tau)^n at a constant acceptance rate."""
    p = VerifyParams()
    tau = float(np.float32(0.1))
    ema = np.array([1.0])
    for n in range(1, 40):
        ema = ov.ema_update(ema, np.array([rho * 4]), np.array([4]), p)
        assert abs(ema[0] - (rho + (1.0 - rho) * (1 - tau) ** n)) < 1e-13


def test_ema_gate_golden():
    """Gate example derived by hand from the page's tau = 0.1, threshold 0.5."""
    with open(os.path.join(GOLDEN, "ema_gate.json")) as f:
        g = json.load(f)
    p = VerifyParams(ema_tau=g["tau"], ema_thresh=g["threshold"])
    for sc in g["scenarios"]:
        ema = np.array([g["ema0"]])
        k_eff_seen = []
        for rate in sc["acceptance_rates"]:
            k_eff = ov.gate_k(np.array([4]), ema, p)
            k_eff_seen.append(int(k_eff[0]))
            ema = ov.ema_update(ema, np.array([round(rate * k_eff[0])]), k_eff, p)
        assert k_eff_seen == sc["expected_k_eff"]


def test_gated_call_has_no_drafts_and_keeps_ema():
    rng = np.random.default_rng(2)
    B, K, V = 8, 4, 16
    logits = rng.normal(size=(B, K + 1, V))
    ema = np.array([0.49, 0.5, 0.51, 0.1, 0.9, 0.499999, 0.5000001, 1.0], dtype=np.float32)
    p = VerifyParams(temperature=1.0, gate_enabled=True, seed=4)
    res = ov.spec_verify(logits, rng.integers(0, V, (B, K)), None, np.full(B, K),
                         np.zeros((B, 1), int), np.zeros(B, int), p, np.full(B, 50), ema)
    off = ema.astype(np.float64) < float(np.float32(0.5))
    assert (res["k_eff"][off] == 0).all() and (res["k_eff"][~off] == K).all()
    assert (res["accept_len"][off] == 0).all()
    np.testing.assert_array_equal(res["ema"][off], ema[off].astype(np.float64))
    np.testing.assert_array_equal(res["kv_len"][off], 50 - K)


def test_kv_len_invariant_and_ranges():
    rng = np.random.default_rng(8)
    B, K, V = 128, 4, 24
    logits = rng.normal(0, 2, size=(B, K + 1, V))
    drafts = np.argmax(logits[:, :K], axis=-1)            # likely accepted
    drafts[::3] = rng.integers(0, V, size=drafts[::3].shape)
    k = rng.integers(0, K + 1, size=B)
    kv = rng.integers(10, 100, size=B)
    res = ov.spec_verify(logits, drafts, None, k, np.zeros((B, 1), int), np.zeros(B, int),
                         VerifyParams(temperature=0.7, gate_enabled=False, seed=1, step=2), kv,
                         np.ones(B))
    a = res["accept_len"]
    assert ((0 <= a) & (a <= k)).all()
    np.testing.assert_array_equal(res["kv_len"], kv - k + a)
    assert ((res["out_tokens"] >= 0).sum(axis=1) == a + 1).all()


def test_point_mass_residual_excludes_the_rejected_draft():
    # a rejected draft can never be re-emitted at the same position
    rng = np.random.default_rng(3)
    B, V = 4000, 6
    logits = np.tile(np.log(np.array([0.3, 0.25, 0.2, 0.1, 0.1, 0.05]))[None, None, :], (B, 2, 1))
    drafts = np.zeros((B, 1), dtype=np.int64)
    res = ov.spec_verify(logits, drafts, None, np.ones(B), np.zeros((B, 1), int), np.zeros(B, int),
                         VerifyParams(temperature=1.0, gate_enabled=False, seed=9), np.zeros(B),
                         np.ones(B), seq_ids=np.arange(B))
    rej = res["accept_len"] == 0
    assert rej.any() and (res["out_tokens"][rej, 0] != 0).all()


def test_invalid_draft_is_rejected():
    logits = np.zeros((1, 2, 8))
    res = ov.spec_verify(logits, np.array([[8]]), None, np.array([1]), np.zeros((1, 1), int),
                         np.zeros(1, int), VerifyParams(temperature=1.0, gate_enabled=False), np.zeros(1),
                         np.ones(1))
    assert res["accept_len"][0] == 0 and 0 <= res["out_tokens"][0, 0] < 8


def _gate_golden():
    with open(os.path.join(GOLDEN, "gate_variants.json")) as f:
        return json.load(f)


def test_gate_reprobe_golden():
    """Re-probing a gated-off sequence every P calls (hand-derived trajectories)."""
    g = _gate_golden()
    for sc in g["probe"]:
        p = VerifyParams(ema_tau=g["tau"], ema_thresh=g["threshold"], probe_interval=sc["probe_interval"])
        ema = np.array([g["ema0"]])
        seen = []
        for step, rate in enumerate(sc["acceptance_rates"]):
            p.step = step
            k_eff = ov.gate_k(np.array([g["k"]]), ema, p)
            seen.append(int(k_eff[0]))
            ema = ov.ema_update(ema, np.array([round(rate * k_eff[0])]), k_eff, p)
        assert seen == sc["expected_k_eff"], (sc, seen)


def test_gate_cooling_golden():
    """No drafts for C calls after a partial acceptance (hand-derived trajectory)."""
    g = _gate_golden()
    for sc in g["cooling"]:
        p = VerifyParams(ema_tau=g["tau"], ema_thresh=g["threshold"], cool_steps=sc["cool_steps"])
        ema, cool = np.array([g["ema0"]]), np.array([0])
        seen, cools = [], []
        for acc in sc["accepted_when_verifying"]:
            k_eff = ov.gate_k(np.array([g["k"]]), ema, p, cool)
            seen.append(int(k_eff[0]))
            a = np.array([acc if k_eff[0] > 0 else 0])
            ema = ov.ema_update(ema, a, k_eff, p)
            cool = ov.cool_update(cool, a, k_eff, p)
            cools.append(int(cool[0]))
        assert seen == sc["expected_k_eff"] and cools == sc["expected_cool_after"], (seen, cools)


def test_gate_variants_through_spec_verify():
    """The variants inside one whole call: a cooling sequence verifies nothing and
    counts down, a probe step opens a gated-off sequence, the rest as before."""
    rng = np.random.default_rng(12)
    B, K, V = 4, 3, 16
    logits = rng.normal(size=(B, K + 1, V)) * 2
    drafts = rng.integers(0, V, (B, K))
    ema = np.array([0.2, 0.2, 0.9, 0.9], dtype=np.float32)
    cool = np.array([0, 3, 1, 0])
    for step, probe in ((8, True), (9, False)):
        p = VerifyParams(temperature=1.0, gate_enabled=True, seed=3, step=step, probe_interval=4, cool_steps=2)
        res = ov.spec_verify(logits, drafts, None, np.full(B, K), np.zeros((B, 1), int), np.zeros(B, int), p,
                             np.full(B, 50), ema, gate_state=cool)
        want = np.array([K if probe else 0, 0, 0, K])
        np.testing.assert_array_equal(res["k_eff"], want)
        assert res["gate_state"][1] == 2 and res["gate_state"][2] == 0
        a = res["accept_len"]
        np.testing.assert_array_equal(res["kv_len"], 50 - K + a)
        part = (a > 0) & (a < want)
        np.testing.assert_array_equal(res["gate_state"][[0, 3]], np.where(part, 2, 0)[[0, 3]])
