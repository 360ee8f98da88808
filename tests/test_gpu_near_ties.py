"""Planted near-ties: every decision that floating point takes is screened
in fp32 with a margin and re-taken in fp64 inside it.  At random inputs
those re-takes run about once per 10^4 rows, so the lockstep cases may never
reach them.  Here each case builds its inputs from the oracle's own noise so
that one decision lies about 5e-5 (in log / score units) from its boundary:

* the accept test u q(d) <= p(d), point mass (the temperature is solved for)
  and dense q (q(d) is set), on both sides of the boundary;
* the top two Gumbel scores of a point-mass residual and of a bonus sample
  (the temperature is solved for), on both sides;
* the dense residual max(0, p - q): a winner whose ln p - ln q is 5e-5, and
  two residual scores 5e-5 apart;
* a greedy argmax tie (two equal logits).

Each GPU result must equal the oracle's element by element (no excuse is
allowed), and the library's diagnostic counter of the planted path must
show that the fp64 re-take ran.  Source of the rules: SwiftLM page,
paragraph on algorithmic equivalence after Leviathan et al."""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from oracle import philox as op
from oracle import verify as ov

pytestmark = pytest.mark.gpu

GAP = 5e-5
SEED, STEP = 77, 5


def _round(x, dtype):
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _run(logits, drafts, q, k, T, dtype, hist=None, lens=None, **kw):
    """GPU and oracle on the same inputs; returns (gpu outputs, oracle result, counters)."""
    B, K1, V = logits.shape
    x = _round(logits, dtype)
    xf = x.float().numpy().astype(np.float64)
    if hist is None:
        hist = np.zeros((B, 1), dtype=np.int64)
        lens = np.zeros(B, dtype=np.int64)
    params = dict(temperature=float(np.float32(T)), gate_enabled=False, seed=SEED, step=STEP, **kw)
    dev = "cuda"
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K1 - 1, V)
    sp.get_status(clear=True)
    sp.get_counters(clear=True)
    pen = kw.get("rep_penalty", 1.0) != 1.0
    sp.spec_verify(x.cuda(), torch.from_numpy(drafts.astype(np.int32)).cuda(),
                   None if q is None else torch.from_numpy(q.astype(np.float32)).cuda(),
                   torch.from_numpy(k.astype(np.int32)).cuda(),
                   torch.from_numpy(hist.astype(np.int32)).cuda() if pen else None,
                   torch.from_numpy(lens.astype(np.int32)).cuda() if pen else None,
                   sp.VerifyParams(**params), kv, ema, out, acc, ws)
    cnt = sp.get_counters(clear=True)
    assert sp.get_status(clear=True) == 0
    res = ov.spec_verify(xf, drafts, None if q is None else q.astype(np.float32), k, hist, lens,
                         ov.VerifyParams(**params), np.full(B, 100), np.ones(B))
    return (out.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy()), res, cnt


def _check_equal(gpu, res):
    out, acc, kv = gpu
    np.testing.assert_array_equal(acc, res["accept_len"])
    np.testing.assert_array_equal(out, res["out_tokens"])
    np.testing.assert_array_equal(kv, res["kv_len"])


def _lp(z_row, T, v):
    """ln p_v of a transformed row at fp32 temperature T (fp64, the oracle's softmax)."""
    return float(ov.log_softmax(z_row / float(np.float32(T)))[v])


# ---------------------------------------------------------------- accept test

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("side", [-1, 1])
def test_accept_point_mass_near_boundary(dtype, side):
    # sequence 0's first draft is its row's largest logit + 1, so ln p(d) falls
    # from 0 towards -ln V as T grows; T is solved so that ln u - ln p(d) = side * GAP
    rng = np.random.default_rng(1 + side)
    B, K, V = 3, 2, 20000
    logits = rng.standard_normal((B, K + 1, V)) * 3
    drafts = rng.integers(0, V, size=(B, K))
    d = int(drafts[0, 0])
    logits[0, 0, d] = logits[0, 0].max() + 1.0
    x = _round(logits, dtype).float().numpy().astype(np.float64)
    z = x[0, 0]
    lnu = float(np.log(op.accept_uniform(SEED, 0, STEP, 1)))
    f = lambda T: lnu - _lp(z, T, d) - side * GAP  # noqa: E731  (increasing in T)
    lo, hi = 0.02, 50.0
    assert f(lo) < 0 < f(hi)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        lo, hi = (mid, hi) if f(mid) < 0 else (lo, mid)
    T = float(np.float32(hi))
    margin = lnu - _lp(z, T, d)
    assert abs(margin - side * GAP) < 5e-6, margin
    k = np.array([1, 2, 2])
    gpu, res, cnt = _run(logits, drafts, None, k, T, dtype)
    _check_equal(gpu, res)
    assert res["accept_len"][0] == (1 if side < 0 else 0)
    assert cnt["accept_f64"] >= 1, cnt


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("side", [-1, 1])
def test_accept_dense_near_boundary(dtype, side):
    # q(d_1) of every sequence set so that ln u + ln q - ln p(d) = side * GAP
    rng = np.random.default_rng(5 + side)
    B, K, V, T = 4, 2, 20000, 0.6
    logits = rng.standard_normal((B, K + 1, V)) * 3
    x = _round(logits, dtype).float().numpy().astype(np.float64)
    q = np.exp(rng.standard_normal((B, K, V)))
    q /= q.sum(-1, keepdims=True)
    drafts = rng.integers(0, V, size=(B, K))
    for b in range(B):
        d = int(drafts[b, 0])
        lnu = float(np.log(op.accept_uniform(SEED, b, STEP, 1)))
        q[b, 0, d] = np.exp(_lp(x[b, 0], T, d) - lnu + side * GAP)
    q = q.astype(np.float32)
    for b in range(B):
        d = int(drafts[b, 0])
        m = np.log(op.accept_uniform(SEED, b, STEP, 1)) + np.log(np.float64(q[b, 0, d])) - _lp(x[b, 0], T, d)
        assert abs(m - side * GAP) < 5e-6
    gpu, res, cnt = _run(logits, drafts, q, np.full(B, K), T, dtype)
    _check_equal(gpu, res)
    if side > 0:
        assert (res["accept_len"] == 0).all()
    else:
        assert (res["accept_len"] >= 1).all()
    assert cnt["accept_f64"] >= B, cnt


# ---------------------------------------------------------------- sampling

def _plant_top2(rng, V, seq, pos, side, hi=40.0, lo_scale=0.5):
    """A row whose two best Gumbel scores differ by side * GAP: returns
    (row, v1, v2, T).  Every other logit is N(0, lo_scale^2), far below."""
    row = rng.standard_normal(V) * lo_scale
    for _ in range(100):
        v1, v2 = (int(v) for v in rng.choice(V, size=2, replace=False))
        lnE1 = float(np.log(op.exp_noise(SEED, seq, STEP, pos, v1)))
        lnE2 = float(np.log(op.exp_noise(SEED, seq, STEP, pos, v2)))
        D = side * GAP + lnE1 - lnE2           # (z1 - z2) / T must equal D
        if abs(D) < 0.05:
            continue
        z1 = hi
        z2 = float(torch.tensor(z1 - D * 1.0).to(torch.bfloat16).float())   # aim at T ~ 1
        if (z1 - z2) * D <= 0:
            continue
        T = float(np.float32((z1 - z2) / D))
        if not 0.5 < T < 1.2:
            continue
        s1 = z1 / np.float64(np.float32(T)) - lnE1
        s2 = z2 / np.float64(np.float32(T)) - lnE2
        if abs((s1 - s2) - side * GAP) < 5e-6:
            row[v1], row[v2] = z1, z2
            return row, v1, v2, T
    raise AssertionError("no pair found")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("side", [-1, 1])
@pytest.mark.parametrize("mode", ["bonus", "point_mass_residual"])
def test_sample_top_two_near_tie(dtype, side, mode):
    rng = np.random.default_rng({"bonus": 11, "point_mass_residual": 13}[mode] + side)
    B, K, V = 2, 1, 20000
    row, v1, v2, T = _plant_top2(rng, V, seq=0, pos=0, side=side)
    logits = rng.standard_normal((B, K + 1, V)) * 0.5
    logits[0, 0] = row
    drafts = np.zeros((B, K), dtype=np.int64)
    if mode == "bonus":
        k = np.array([0, 1])
    else:
        drafts[0, 0] = int(np.argmin(row))     # p(d) ~ e^-40: rejected
        k = np.array([1, 1])
    gpu, res, cnt = _run(logits, drafts, None, k, T, dtype)
    _check_equal(gpu, res)
    assert res["accept_len"][0] == 0
    assert res["out_tokens"][0, 0] == (v1 if side > 0 else v2)
    assert res["sample_margin"][0] < 1e-4
    assert cnt["sample_f64"] >= 1, cnt


def test_sample_top_two_near_tie_softcap_penalty():
    # the same with a soft cap and a repetition penalty (v1 in the window):
    # the pair is planted on the transformed values
    rng = np.random.default_rng(17)
    B, K, V, cap, r = 1, 0, 20000, 50.0, 1.3
    hist = rng.integers(0, V, size=(B, 40))
    lens = np.full(B, 40)
    for _ in range(50):
        base = rng.standard_normal(V) * 0.5
        v1, v2 = (int(v) for v in rng.choice(V, size=2, replace=False))
        hist[0, -1] = v1
        if v2 in hist[0, -16:]:
            continue
        lnE1 = float(np.log(op.exp_noise(SEED, 0, STEP, 0, v1)))
        lnE2 = float(np.log(op.exp_noise(SEED, 0, STEP, 0, v2)))
        D = GAP + lnE1 - lnE2
        if abs(D) < 0.05:
            continue
        x1 = 60.0
        z1 = cap * np.tanh(np.float64(np.float32(x1)) / cap) / r     # penalised (positive)
        z2_want = z1 - D * 0.7
        if not 0 < z2_want < cap * 0.9:
            continue
        x2 = float(np.float32(cap * np.arctanh(z2_want / cap)))
        z2 = cap * np.tanh(np.float64(np.float32(x2)) / cap)
        T = float(np.float32((z1 - z2) / D))
        if not 0.4 < T < 1.0:
            continue
        Tf = np.float64(np.float32(T))
        if abs((z1 / Tf - lnE1) - (z2 / Tf - lnE2) - GAP) > 5e-6:
            continue
        base[v1], base[v2] = x1, x2
        logits = base[None, None, :]
        kw = dict(softcap=cap, rep_penalty=r, rep_window=16)
        gpu, res, cnt = _run(logits, np.zeros((B, 0), dtype=np.int64), None, np.zeros(B, dtype=np.int64), T, "f32",
                             hist=hist, lens=lens, **kw)
        _check_equal(gpu, res)
        assert res["out_tokens"][0, 0] == v1 and res["sample_margin"][0] < 1e-4
        assert cnt["sample_f64"] >= 1, cnt
        return
    raise AssertionError("no pair found")


# ---------------------------------------------------------------- dense residual

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dense_residual_winner_barely_positive(dtype):
    # row 0's draft has q = 1 and a tiny p (rejected); the residual is positive
    # only at v1, where ln p - ln q = GAP: below the fp32 decision's 1e-4 guard
    rng = np.random.default_rng(23)
    B, K, V, T = 3, 1, 20000, 0.7
    logits = rng.standard_normal((B, K + 1, V)) * 2
    x = _round(logits, dtype).float().numpy().astype(np.float64)
    q = np.zeros((B, K, V))
    drafts = np.zeros((B, K), dtype=np.int64)
    for b in range(B):
        lp = ov.log_softmax(x[b, 0] / np.float64(np.float32(T)))
        v1 = int(np.argmax(x[b, 0]))
        q[b, 0] = np.exp(lp) * 1.01            # no residual anywhere ...
        q[b, 0, v1] = np.exp(lp[v1] - GAP)     # ... but a sliver at v1
        drafts[b, 0] = int(np.argmin(x[b, 0]))
        q[b, 0, drafts[b, 0]] = 1.0
    q = q.astype(np.float32)
    gpu, res, cnt = _run(logits, drafts, q, np.full(B, K), T, dtype)
    _check_equal(gpu, res)
    assert (res["accept_len"] == 0).all()
    assert cnt["residual_f64"] >= B, cnt


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("side", [-1, 1])
def test_dense_residual_top_two_near_tie(dtype, side):
    # v1 (q = 0) and v2 (q set) have residual scores ln(p - q) - ln E that
    # differ by side * GAP; every other id has q > p
    rng = np.random.default_rng(29 + side)
    B, K, V, T = 2, 1, 20000, 0.8
    logits = rng.standard_normal((B, K + 1, V)) * 2
    drafts = np.zeros((B, K), dtype=np.int64)
    for b in range(B):
        v1, v2 = (int(v) for v in rng.choice(V, size=2, replace=False))
        logits[b, 0, v1] = logits[b, 0, v2] = logits[b, 0].max() + 2.0
        drafts[b, 0] = int(np.argmin(logits[b, 0]))
    x = _round(logits, dtype).float().numpy().astype(np.float64)
    q = np.zeros((B, K, V))
    winners = []
    for b in range(B):
        top = np.argsort(-x[b, 0])[:2]
        lp = ov.log_softmax(x[b, 0] / np.float64(np.float32(T)))
        E = {int(v): float(op.exp_noise(SEED, b, STEP, 0, int(v))) for v in top}
        v2, v1 = sorted(E, key=lambda v: E[v])   # v2 has the smaller E (the larger -ln E)
        q[b, 0] = np.exp(lp) * 1.01
        q[b, 0, v1] = 0.0
        s1 = lp[v1] - np.log(E[v1])
        r2 = np.exp(s1 - side * GAP + np.log(E[v2]))    # s1 - s2 = side * GAP
        assert r2 < np.exp(lp[v2])
        q[b, 0, v2] = np.exp(lp[v2]) - r2
        q[b, 0, drafts[b, 0]] = 1.0
        winners.append(v1 if side > 0 else v2)
    q = q.astype(np.float32)
    gpu, res, cnt = _run(logits, drafts, q, np.full(B, K), T, dtype)
    _check_equal(gpu, res)
    assert (res["accept_len"] == 0).all()
    assert list(res["out_tokens"][:, 0]) == winners
    assert (res["sample_margin"] < 1e-4).all()
    assert cnt["residual_f64"] >= B, cnt


# ---------------------------------------------------------------- greedy

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_greedy_exact_tie_takes_the_lower_id(dtype):
    rng = np.random.default_rng(31)
    B, K, V = 3, 2, 20000
    logits = rng.standard_normal((B, K + 1, V)) * 2
    drafts = rng.integers(0, V, size=(B, K))
    for b in range(B):
        v1, v2 = sorted(int(v) for v in rng.choice(V, size=2, replace=False))
        logits[b, 0, v1] = logits[b, 0, v2] = logits[b, 0].max() + 1.0
        drafts[b, 0] = v2 if b == 0 else v1     # sequence 0 drafts the higher id: rejected
    gpu, res, cnt = _run(logits, drafts, None, np.full(B, K), 0.0, dtype)
    _check_equal(gpu, res)
    assert res["accept_len"][0] == 0 and res["accept_len"][1] >= 1
    assert cnt["greedy_f64"] >= B, cnt
