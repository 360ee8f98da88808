"""Verify / sample / epilogue of one speculative step, in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What one call computes, for every sequence b of a batch (rows j = 0..K of
``logits[b]`` are the target's next-token logits after history ++ d_1..d_j):

1. Row transform (``transform_rows``): Gemma logit soft cap c*tanh(x/c)
   (AX Engine page, "Supported Model Families" table: "logit soft cap"),
   then the repetition penalty (SwiftLM page, M1 Ultra benchmark paragraph:
   ``--repeat-penalty 1.1``), then temperature (same paragraph: 0.6).
2. Target probabilities p_j = softmax(x_j / T) (exact two-pass log-sum-exp).
3. EMA gate (AX Engine page, "Core Technical Architecture & Methods":
   EMA acceptance-rate gating, tau = 0.1, threshold 0.5, disables
   speculation when quality drops): k_eff = k if the gate is off or
   ema >= threshold, else 0.
4. Accept test (SwiftLM page, paragraph on algorithmic equivalence after
   Leviathan et al.: accept with P_target / P_draft): draft i is accepted iff
   u_i * q(d_i) <= p(d_i); the first rejection ends the scan; a = number
   accepted.  At T = 0 (greedy, SwiftLM's DFlash warning paragraph): accept
   iff d_i is the argmax of its row.
5. Sample at row a: on a rejection, from the normalised residual
   max(0, p_a - q_a) (same paragraph: "resample from the corrected
   distribution"); when all drafts are accepted, the bonus token from p_a.
   Sampling is Gumbel-max: argmax_v (log w_v + g_v), which needs no prefix
   sum.  At T = 0 the sample is the argmax.
6. Epilogue (AX Engine page, same section: O(1) rollback by moving the
   sequence-length pointer): out_tokens = d_1..d_a, y, then -1;
   accept_len = a; kv_len <- kv_len - k + a; if k_eff > 0,
   ema <- (1 - tau) * ema + tau * a / k_eff.

Readings where the pages are silent (the same readings hold in the GPU library):
* processors apply in the order soft cap -> penalty -> temperature;
* the penalty divides positive logits by r and multiplies negative ones by
  r, once per distinct id, over the last ``rep_window`` tokens of
  history ++ d_1..d_j for row j (what plain decoding would see there);
* a point-mass draft has q = one-hot(d), so the residual is p with d removed;
* an all-zero residual falls back to sampling from p;
* a draft id outside [0, V) is rejected and the residual is p (no id removed);
* the gate is checked before the update; a gated call has a = 0 and leaves
  the EMA unchanged; the initial EMA is chosen by the caller (1.0 in all
  workloads here);
* all scalar parameters are fp32 values, widened to fp64 here.

Pinned by: tests/test_oracle_verify.py (greedy against an independent
argmax-matching function; closed forms of each processor; EMA closed form;
kv_len invariant), tests/test_oracle_enumeration.py (exact V = 8, K <= 3
enumeration of the emitted-token law for point-mass and dense drafts,
using the rule functions below), tests/test_oracle_chisq.py (V = 32
chi-square of the whole procedure over 10**6 seeded steps, Gumbel-max vs
softmax, and the sample-and-match cross-check).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import philox


@dataclass
class VerifyParams:
    """Scalar knobs of one verify call (fp32 values, as the library takes them)."""
    temperature: float = 1.0
    softcap: float = 0.0
    rep_penalty: float = 1.0
    rep_window: int = 0
    ema_tau: float = 0.1
    ema_thresh: float = 0.5
    gate_enabled: bool = True
    seed: int = 0
    step: int = 0
    probe_interval: int = 0   # > 0: a gated-off sequence verifies on calls with step % interval == 0
    cool_steps: int = 0       # > 0: after a partial acceptance, no drafts for this many calls

    def f64(self, name: str) -> float:
        return float(np.float32(getattr(self, name)))


# ---------------------------------------------------------------- processors

def softcap(x: np.ndarray, c: float) -> np.ndarray:
    """Gemma's logit soft cap c * tanh(x / c); c <= 0 leaves x unchanged."""
    if c <= 0.0:
        return x
    return c * np.tanh(x / c)


def penalty_ids(history_b: np.ndarray, lens_b: int, drafts_b: np.ndarray, j: int,
                window: int) -> np.ndarray:
    """Distinct ids among the last ``window`` tokens of history[:lens] ++ d_1..d_j."""
    if window <= 0:
        return np.zeros(0, dtype=np.int64)
    seq = np.concatenate([np.asarray(history_b[:lens_b], dtype=np.int64),
                          np.asarray(drafts_b[:j], dtype=np.int64)])
    return np.unique(seq[-window:])


def repetition_penalty(x: np.ndarray, ids: np.ndarray, r: float) -> np.ndarray:
    """Penalise each distinct id once: x / r where x > 0, x * r otherwise."""
    if r == 1.0 or ids.size == 0:
        return x
    x = x.copy()
    ids = ids[(ids >= 0) & (ids < x.shape[-1])]
    v = x[ids]
    x[ids] = np.where(v > 0.0, v / r, v * r)
    return x


def transform_rows(logits: np.ndarray, params: VerifyParams, history: np.ndarray,
                   lens: np.ndarray, drafts: np.ndarray) -> np.ndarray:
    """Soft cap then repetition penalty on every row; returns fp64 [B, K+1, V].

    Temperature is applied by the caller (T = 0 means greedy and has no
    division).
    """
    z = softcap(np.asarray(logits, dtype=np.float64), params.f64("softcap"))
    r = params.f64("rep_penalty")
    if r != 1.0 and params.rep_window > 0:
        z = z.copy()
        B, K1, _ = z.shape
        for b in range(B):
            for j in range(K1):
                ids = penalty_ids(history[b], int(lens[b]), drafts[b], j, params.rep_window)
                z[b, j] = repetition_penalty(z[b, j], ids, r)
    return z


def log_softmax(y: np.ndarray) -> np.ndarray:
    """log p = y - logsumexp(y) along the last axis, two-pass and exact in fp64."""
    m = np.max(y, axis=-1, keepdims=True)
    return y - (m + np.log(np.sum(np.exp(y - m), axis=-1, keepdims=True)))


# ---------------------------------------------------------------- rules

def gate_k(k: np.ndarray, ema: np.ndarray, params: VerifyParams, cool=None) -> np.ndarray:
    """Drafts verified this call.

    EMA gate (AX Engine page, "Core Technical Architecture & Methods":
    speculation is disabled when the acceptance EMA drops below the
    threshold): k_eff = k when the gate is disabled or ema >= threshold,
    else 0.  Variants (same page, "Performance Evidence & Results", note
    under the decode table: speculation "cools after partial acceptance";
    and the re-opening of a disabled gate, which the page leaves open):
      * re-probe: with probe_interval P > 0, a gated-off sequence verifies
        its drafts anyway on the calls whose step is a multiple of P (the
        update of that call can re-open the gate);
      * cooling: a sequence whose cooling count (``cool``) is positive
        verifies no drafts this call, whatever the gate says.
    """
    k = np.asarray(k, dtype=np.int64)
    keff = k
    if params.gate_enabled:
        on = np.asarray(ema, dtype=np.float64) >= params.f64("ema_thresh")
        if params.probe_interval > 0 and int(params.step) % int(params.probe_interval) == 0:
            on = np.ones_like(on)
        keff = np.where(on, k, 0)
    if cool is not None and params.cool_steps > 0:
        keff = np.where(np.asarray(cool) > 0, 0, keff)
    return keff


def cool_update(cool, a, k_eff, params: VerifyParams):
    """Cooling count after a call: a cooling sequence counts down; otherwise a
    partial acceptance (0 < a < k_eff) starts cool_steps calls without drafts."""
    cool = np.asarray(cool, dtype=np.int64)
    a = np.asarray(a, dtype=np.int64)
    k_eff = np.asarray(k_eff, dtype=np.int64)
    partial = (a > 0) & (a < k_eff)
    return np.where(cool > 0, cool - 1, np.where(partial, int(params.cool_steps), 0))


def accept_draft(u, p_d, q_d):
    """Leviathan/Chen test: accept iff u * q(d) <= p(d) (so q(d) = 0 accepts)."""
    return np.asarray(u) * np.asarray(q_d) <= np.asarray(p_d)


def residual_weights(p_row: np.ndarray, q_row: np.ndarray) -> np.ndarray:
    """Unnormalised corrected distribution max(0, p - q)."""
    return np.maximum(0.0, p_row - q_row)


def gumbel_argmax(log_w: np.ndarray, g: np.ndarray):
    """argmax_v (log w_v + g_v) along the last axis, lowest id on ties.

    Entries with log w = -inf (zero weight) can never win.  Returns the ids
    and the gap between the best and second-best scores (the margin that
    decides whether a near-tie may be excused).
    """
    s = log_w + g
    y = np.argmax(s, axis=-1)
    top = np.take_along_axis(s, y[..., None], axis=-1)[..., 0]
    s2 = s.copy()
    np.put_along_axis(s2, y[..., None], -np.inf, axis=-1)
    gap = top - np.max(s2, axis=-1)
    return y, gap


def ema_update(ema: np.ndarray, a: np.ndarray, k_eff: np.ndarray, params: VerifyParams):
    """ema <- (1 - tau) * ema + tau * a / k_eff on calls with k_eff > 0."""
    tau = params.f64("ema_tau")
    ema = np.asarray(ema, dtype=np.float64)
    k_eff = np.asarray(k_eff, dtype=np.int64)
    rate = np.where(k_eff > 0, np.asarray(a, dtype=np.float64) / np.maximum(k_eff, 1), 0.0)
    return np.where(k_eff > 0, (1.0 - tau) * ema + tau * rate, ema)


# ---------------------------------------------------------------- one call

def spec_verify(logits, drafts, draft_probs, k, history, lens, params: VerifyParams,
                kv_len, ema, seq_ids=None, gate_state=None):
    """One verify call over a batch; returns outputs plus diagnostics.

    logits       [B, K+1, V]  target logits (any float dtype, widened to fp64)
    drafts       [B, K]       draft ids d_1..d_K (entries beyond k[b] unused)
    draft_probs  [B, K, V] or None (None: point-mass drafts, q = one-hot(d))
    k            [B]          number of drafts to verify per sequence
    history      [B, Lcap], lens [B]: for the repetition-penalty window
    kv_len [B], ema [B]: state before the call
    seq_ids      [B]          the sequence ids that key the noise (default 0..B-1)
    gate_state   [B] or None  cooling counts before the call (used when cool_steps > 0)

    Returns a dict with out_tokens [B, K+1], accept_len [B], kv_len [B],
    ema [B] (fp64), k_eff [B] and the margins used by the parity harness:
    accept_margin [B, K] (|ln u + ln q - ln p| of each test made, else inf),
    sample_margin [B] (gap of the top two sampling scores), ema_margin [B].
    """
    logits = np.asarray(logits)
    B, K1, V = logits.shape
    K = K1 - 1
    drafts = np.asarray(drafts, dtype=np.int64).reshape(B, K)
    k = np.asarray(k, dtype=np.int64)
    seq_ids = np.arange(B, dtype=np.int64) if seq_ids is None else np.asarray(seq_ids, dtype=np.int64)
    T = params.f64("temperature")
    greedy = T == 0.0
    dense = draft_probs is not None

    cool = np.zeros(B, dtype=np.int64) if gate_state is None else np.asarray(gate_state, dtype=np.int64)
    k_eff = gate_k(k, ema, params, cool if params.cool_steps > 0 else None)
    z = transform_rows(logits, params, history, lens, drafts)
    rows = np.arange(B)

    accepting = np.ones(B, dtype=bool)
    a = np.zeros(B, dtype=np.int64)
    accept_margin = np.full((B, K), np.inf)
    if greedy:
        arg = np.argmax(z, axis=-1)                     # [B, K+1], lowest id on ties
    else:
        logp = log_softmax(z / T)                       # [B, K+1, V]

    for i in range(1, K + 1):
        live = accepting & (i <= k_eff)
        if not live.any():
            break
        d = drafts[:, i - 1]
        valid = (d >= 0) & (d < V)
        dc = np.clip(d, 0, V - 1)
        if greedy:
            zi = z[rows, i - 1]
            acc = valid & (dc == arg[:, i - 1])
            others = zi.copy()
            others[rows, dc] = -np.inf
            margin = np.abs(zi[rows, dc] - np.max(others, axis=-1))
        else:
            lp = logp[rows, i - 1, dc]
            q = draft_probs[rows, i - 1, dc].astype(np.float64) if dense else np.ones(B)
            u = philox.accept_uniform(params.seed, seq_ids, params.step, i)
            acc = valid & accept_draft(u, np.exp(lp), q)
            with np.errstate(divide="ignore"):
                margin = np.abs(np.log(u) + np.log(q) - lp)
        accept_margin[live, i - 1] = np.where(valid, margin, np.inf)[live]
        a = np.where(live & acc, i, a)
        accepting = live & acc

    # sample at row a: residual on a rejection, bonus when all k_eff accepted
    if greedy:
        y = arg[rows, a]
        za = z[rows, a]
        s2 = za.copy()
        s2[rows, y] = -np.inf
        sample_margin = za[rows, y] - np.max(s2, axis=-1)
    else:
        lpa = logp[rows, a]                             # [B, V]
        pa = np.exp(lpa)
        rejected = a < k_eff
        da = drafts[rows, np.minimum(a, K - 1)] if K > 0 else np.zeros(B, dtype=np.int64)
        da_valid = rejected & (da >= 0) & (da < V)
        if dense:
            qa = draft_probs[rows, np.minimum(a, K - 1)].astype(np.float64) if K > 0 else np.zeros_like(pa)
            qa = np.where(da_valid[:, None], qa, 0.0)
        else:
            qa = np.zeros_like(pa)
            qa[rows[da_valid], da[da_valid]] = 1.0
        w = np.where(rejected[:, None], residual_weights(pa, qa), pa)
        empty = ~(w > 0.0).any(axis=-1)
        w = np.where(empty[:, None], pa, w)             # all-zero residual: sample from p
        with np.errstate(divide="ignore"):
            log_w = np.log(w)
        g = philox.gumbel_row(params.seed, seq_ids, params.step, a, V)
        y, sample_margin = gumbel_argmax(log_w, g)

    cols = np.arange(K + 1)[None, :]
    padded = np.concatenate([drafts, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    out = np.where(cols < a[:, None], padded, -1)
    out[rows, a] = y
    ema_new = ema_update(ema, a, k_eff, params)
    thresh = params.f64("ema_thresh")
    return {
        "gate_state": cool_update(cool, a, k_eff, params) if params.cool_steps > 0 else cool,
        "out_tokens": out,
        "accept_len": a,
        "kv_len": np.asarray(kv_len, dtype=np.int64) - k + a,
        "ema": ema_new,
        "k_eff": k_eff,
        "accept_margin": accept_margin,
        "sample_margin": sample_margin,
        "ema_margin": np.abs(np.asarray(ema, dtype=np.float64) - thresh),
    }
