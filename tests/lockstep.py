"""Lockstep parity harness: the CUDA library against the fp64 oracle.

Both sides start from the same seeded inputs.  Every step the oracle runs on
its OWN state (history, lengths, kv_len, EMA), never on values the GPU
produced; the GPU state is compared with it:

* drafts, draft counts, accept lengths, kv_len and tokens: bit-exact;
* EMA: |difference| <= 1e-6;
* a token / accept length may differ only where the oracle's margin (gap of
  the top two sampling scores, or |ln u + ln q - ln p| of the accept test)
  is below 1e-4, or an EMA gate flip where |ema - threshold| < 1e-6; such
  excused rows must be at most 1e-5 of all rows.  After an excused
  mismatch the GPU state is overwritten with the oracle's (uploaded), so the
  trajectories never diverge.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from oracle import ngram as on
from oracle import verify as ov
from speculative_decoding_draft_ngram_gb300 import workloads as wl

MARGIN = 1e-4
EMA_TOL = 1e-6
EXCUSE_RATE = 1e-5


@dataclass
class Report:
    steps: int = 0
    rows: int = 0
    rows_read: int = 0
    excused: int = 0
    accepted: int = 0
    drafted: int = 0
    gated: int = 0
    accept_hist: list = field(default_factory=list)   # counts of accept length a = 0, 1, ... (oracle side)
    notes: list = field(default_factory=list)

    def count_accepts(self, a):
        for v in np.asarray(a).ravel().tolist():
            while len(self.accept_hist) <= v:
                self.accept_hist.append(0)
            self.accept_hist[v] += 1

    def tokens_per_sequence_step(self) -> float:
        n = sum(self.accept_hist)
        return sum((i + 1) * c for i, c in enumerate(self.accept_hist)) / n if n else 0.0


GATE_KEYS = ("probe_interval", "cool_steps")


def _oracle_params(cfg: wl.Config, T: float, step: int, seed: int, **var) -> ov.VerifyParams:
    return ov.VerifyParams(temperature=T, softcap=cfg.softcap, rep_penalty=cfg.rep_penalty,
                           rep_window=cfg.rep_window, gate_enabled=cfg.gate, seed=seed, step=step,
                           **{k: v for k, v in var.items() if k in GATE_KEYS})


def _gpu_params(cfg: wl.Config, T: float, step: int, seed: int, **var) -> sp.VerifyParams:
    return sp.VerifyParams(temperature=T, softcap=cfg.softcap, rep_penalty=cfg.rep_penalty,
                           rep_window=cfg.rep_window, gate_enabled=cfg.gate, seed=seed, step=step, **var)


def oracle_verify(logits, drafts, q, k, hist, lens, params, kv, ema, chunk=16, gate_state=None):
    """The oracle's verify over the batch, in chunks of sequences (same result)."""
    B = logits.shape[0]
    parts = []
    for lo in range(0, B, chunk):
        hi = min(B, lo + chunk)
        parts.append(ov.spec_verify(logits[lo:hi].astype(np.float64), drafts[lo:hi],
                                    None if q is None else q[lo:hi], k[lo:hi], hist[lo:hi], lens[lo:hi],
                                    params, kv[lo:hi], ema[lo:hi], seq_ids=np.arange(lo, hi),
                                    gate_state=None if gate_state is None else gate_state[lo:hi]))
    return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}


def compare(step, a_g, t_g, kv_gh, ema_gh, res, rep: Report, ids=None):
    """Compare one step's GPU outputs with the oracle's (rows of the same
    sequences); raise on a mismatch that the margin rule does not excuse.
    Returns the mask of (excused) mismatching sequences."""
    a_o = res["accept_len"]
    t_o = res["out_tokens"]
    bad = (a_g != a_o) | (t_g != t_o).any(axis=1) | (kv_gh != res["kv_len"]) | \
          (np.abs(ema_gh - res["ema"]) > EMA_TOL)
    for b in np.nonzero(bad)[0]:
        excusable = False
        if a_g[b] != a_o[b]:
            i = min(a_g[b], a_o[b])
            excusable = res["accept_margin"][b, i] < MARGIN
        elif (t_g[b] != t_o[b]).any():
            excusable = res["sample_margin"][b] < MARGIN
        if res["ema_margin"][b] < EMA_TOL:
            excusable = True
        sb = b if ids is None else int(ids[b])
        msg = (f"step {step} seq {sb}: gpu a={a_g[b]} tok={t_g[b].tolist()} kv={kv_gh[b]} ema={ema_gh[b]!r}; "
               f"oracle a={a_o[b]} tok={t_o[b].tolist()} kv={res['kv_len'][b]} ema={res['ema'][b]!r} "
               f"acc_margin={res['accept_margin'][b].tolist()} sample_margin={res['sample_margin'][b]!r}")
        assert excusable, "parity failure: " + msg
        rep.excused += 1
        rep.notes.append(msg)
    return bad


def run_sampled(cfg: wl.Config, steps: int, sample: int, T: float | None = None, device="cuda",
                seed: int | None = None, ema0: float = 1.0, **sched) -> Report:
    """Full-size steps on the GPU (the whole batch, in the launch configuration
    the benchmark uses); the oracle checks a seeded sample of ``sample``
    sequences one by one (sequences are independent; their Philox streams are
    keyed by their own index)."""
    T = cfg.temperature if T is None else T
    seed = cfg.sampler_seed if seed is None else seed
    rep = Report()
    B, K, V = cfg.B, cfg.K, cfg.V
    hist_full, lens_full = wl.histories(cfg, "cpu")
    ids = np.sort(np.random.default_rng(cfg.data_seed).choice(B, size=min(sample, B), replace=False))
    hist_o = hist_full.numpy()[ids].astype(np.int64)
    lens_o = lens_full.numpy()[ids].astype(np.int64)
    hist_g = hist_full.to(device)
    lens_g = lens_full.to(device)
    ema_o = np.full(len(ids), float(np.float32(ema0)), dtype=np.float64)
    ema_g = torch.full((B,), float(np.float32(ema0)), dtype=torch.float32, device=device)
    kv_g = lens_g.clone()
    use_ngram = not cfg.dense
    table = stats = None
    if use_ngram:
        table = sp.NgramTable(B, V, B * cfg.hist_cap, device=device)
        sp.ngram_update(table, hist_g, lens_g)
        stats = [on.continuation_stats(hist_o[i], int(lens_o[i])) for i in range(len(ids))]
    ws = sp.spec_verify_workspace(B, K, V, device)
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=device)
    out_acc = torch.empty((B,), dtype=torch.int32, device=device)
    g = wl._gen(cfg.data_seed + 1, "cpu")
    bprob = wl.boost_probs(cfg, "cpu")
    zcdf = wl.zipf_cdf(cfg.zipf_ids or cfg.V, cfg.zipf_s)
    sp.get_status(clear=True)
    for step in range(steps):
        limits = wl.draft_limits(cfg, g, "cpu")
        fb = wl.fallback_drafts(cfg, g, "cpu", zcdf)
        logits = wl.step_logits(cfg, g, device="cpu")
        if use_ngram:
            d_g, k_g = sp.ngram_draft(table, hist_g, lens_g, K, k_limit=limits.to(device),
                                      fallback=None if fb is None else fb.to(device))
            d_o, k_o = on.draft_batch(hist_o, lens_o, K, k_limit=limits.numpy()[ids], stats=stats,
                                      fallback=None if fb is None else fb.numpy()[ids])
            d_gh, k_gh = d_g.cpu().numpy(), k_g.cpu().numpy()
            assert np.array_equal(k_gh[ids], k_o), f"step {step}: draft counts differ"
            assert np.array_equal(d_gh[ids], d_o), f"step {step}: drafts differ"
            drafts, k, q = torch.from_numpy(d_gh), torch.from_numpy(k_gh), None
        else:
            q, drafts = wl.dense_draft(cfg, logits, g)
            k = torch.full((B,), K, dtype=torch.int32)
        logits = wl.apply_boost(cfg, logits, drafts, k, bprob, g)
        kv_all = lens_g.cpu().numpy().astype(np.int64) + k.numpy()
        kv_g.copy_(torch.from_numpy(kv_all.astype(np.int32)))
        sp.spec_verify(logits.to(device), drafts.to(device), None if q is None else q.to(device), k.to(device),
                       hist_g, lens_g, _gpu_params(cfg, T, step, seed, **sched), kv_g, ema_g, out_tok, out_acc, ws)
        res = ov.spec_verify(logits[ids].double().numpy(), drafts.numpy()[ids].astype(np.int64),
                             None if q is None else q[ids].numpy(), k.numpy()[ids].astype(np.int64), hist_o,
                             lens_o, _oracle_params(cfg, T, step, seed), kv_all[ids],
                             ema_o.astype(np.float32), seq_ids=ids)
        a_g = out_acc.cpu().numpy()[ids]
        t_g = out_tok.cpu().numpy()[ids]
        kv_gh = kv_g.cpu().numpy()[ids]
        ema_gh = ema_g.cpu().numpy()[ids].astype(np.float64)
        rep.rows += len(ids) * (K + 1)
        rep.rows_read += int((res["k_eff"] + 1).sum())
        rep.accepted += int(res["accept_len"].sum())
        rep.drafted += int(res["k_eff"].sum())
        rep.count_accepts(res["accept_len"])
        bad = compare(step, a_g, t_g, kv_gh, ema_gh, res, rep, ids)
        sp.spec_append(hist_g, lens_g, out_tok, out_acc)
        for i in range(len(ids)):
            a = int(res["accept_len"][i])
            hist_o[i, lens_o[i]:lens_o[i] + a + 1] = res["out_tokens"][i, :a + 1]
            if stats is not None:
                on.extend_stats(stats[i], hist_o[i], int(lens_o[i]), int(lens_o[i]) + a + 1)
            lens_o[i] += a + 1
        ema_o = res["ema"].astype(np.float32).astype(np.float64)
        if bad.any():  # put the oracle's state into the sampled sequences
            h = hist_g.cpu()
            h[torch.from_numpy(ids)] = torch.from_numpy(hist_o.astype(np.int32))
            hist_g.copy_(h)
            ln = lens_g.cpu()
            ln[torch.from_numpy(ids)] = torch.from_numpy(lens_o.astype(np.int32))
            lens_g.copy_(ln)
            e = ema_g.cpu()
            e[torch.from_numpy(ids)] = torch.from_numpy(ema_o.astype(np.float32))
            ema_g.copy_(e)
            if use_ngram:
                table.reset()
        else:
            assert np.array_equal(lens_g.cpu().numpy()[ids], lens_o)
        if use_ngram:
            sp.ngram_update(table, hist_g, lens_g)
        rep.steps += 1
    status = sp.get_status(clear=True)
    assert status == 0, f"device status bits set: {sp.status_names(status)}"
    assert rep.excused <= EXCUSE_RATE * rep.rows, \
        f"{rep.excused} excused rows out of {rep.rows} exceed 1e-5:\n" + "\n".join(rep.notes)
    if table is not None:
        table.close()
    return rep


def run(cfg: wl.Config, steps: int, T: float | None = None, device="cuda", seed: int | None = None,
        oracle_chunk: int = 16, ema0: float = 1.0, min_count: int = 1, **sched) -> Report:
    """Run ``steps`` lockstep steps of cfg; raise AssertionError on a parity failure.
    ``sched``: schedule / early_exit of the GPU calls (the outputs must not depend on
    them) and the gate variants probe_interval / cool_steps (on both sides; the
    cooling counts are compared bit-exact every step); ``min_count``: the n-gram
    evidence threshold of the drafts (both sides)."""
    T = cfg.temperature if T is None else T
    seed = cfg.sampler_seed if seed is None else seed
    rep = Report()
    hist_o, lens_o = wl.histories(cfg, "cpu")
    hist_o = hist_o.numpy().astype(np.int64)
    lens_o = lens_o.numpy().astype(np.int64)
    B, K, V = cfg.B, cfg.K, cfg.V
    hist_g = torch.from_numpy(hist_o.astype(np.int32)).to(device)
    lens_g = torch.from_numpy(lens_o.astype(np.int32)).to(device)
    ema_o = np.full(B, float(np.float32(ema0)), dtype=np.float64)
    ema_g = torch.full((B,), float(np.float32(ema0)), dtype=torch.float32, device=device)
    kv_o = lens_o.copy()
    kv_g = torch.from_numpy(kv_o.astype(np.int32)).to(device)
    use_ngram = not cfg.dense
    table = None
    stats = None
    if use_ngram:
        table = sp.NgramTable(B, V, B * cfg.hist_cap, device=device)
        if min_count != 1:
            table.set_min_count(min_count)
        sp.ngram_update(table, hist_g, lens_g)
        stats = [on.continuation_stats(hist_o[b], int(lens_o[b])) for b in range(B)]
    ws = sp.spec_verify_workspace(B, K, V, device)
    cooling = sched.get("cool_steps", 0) > 0
    cool_o = np.zeros(B, dtype=np.int64)
    cool_g = torch.zeros(B, dtype=torch.int32, device=device) if cooling else None
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=device)
    out_acc = torch.empty((B,), dtype=torch.int32, device=device)
    g = wl._gen(cfg.data_seed + 1, "cpu")
    bprob = wl.boost_probs(cfg, "cpu")
    zcdf = wl.zipf_cdf(cfg.zipf_ids or cfg.V, cfg.zipf_s)
    sp.get_status(clear=True)

    for step in range(steps):
        limits = wl.draft_limits(cfg, g, "cpu")
        fb = wl.fallback_drafts(cfg, g, "cpu", zcdf)
        logits = wl.step_logits(cfg, g, device="cpu")
        # ---- drafts
        if use_ngram:
            d_o, k_o = on.draft_batch(hist_o, lens_o, K, k_limit=limits.numpy(), stats=stats,
                                      fallback=None if fb is None else fb.numpy(), min_count=min_count)
            d_g, k_g = sp.ngram_draft(table, hist_g, lens_g, K, k_limit=limits.to(device),
                                      fallback=None if fb is None else fb.to(device))
            d_g_h, k_g_h = d_g.cpu().numpy(), k_g.cpu().numpy()
            assert np.array_equal(k_g_h, k_o), f"step {step}: draft counts differ\n{k_g_h}\n{k_o}"
            assert np.array_equal(d_g_h, d_o), f"step {step}: drafts differ\n{d_g_h}\n{d_o}"
            drafts = torch.from_numpy(d_o.astype(np.int32))
            k = torch.from_numpy(k_o.astype(np.int32))
            q = None
        else:
            q, drafts = wl.dense_draft(cfg, logits, g)
            k = torch.full((B,), K, dtype=torch.int32)
        logits = wl.apply_boost(cfg, logits, drafts, k, bprob, g)
        # the verify forward wrote k + 1 positions after the committed ones
        kv_o = lens_o - 1 + k.numpy() + 1
        kv_g.copy_(torch.from_numpy(kv_o.astype(np.int32)))
        # ---- verify on both sides
        res = oracle_verify(logits.float().numpy(), drafts.numpy().astype(np.int64),
                            None if q is None else q.numpy(), k.numpy().astype(np.int64), hist_o, lens_o,
                            _oracle_params(cfg, T, step, seed, **sched), kv_o, ema_o.astype(np.float32), oracle_chunk,
                            gate_state=cool_o)
        sp.spec_verify(logits.to(device), drafts.to(device), None if q is None else q.to(device), k.to(device),
                       hist_g, lens_g, _gpu_params(cfg, T, step, seed, gate_state=cool_g, **sched), kv_g, ema_g,
                       out_tok, out_acc, ws)
        a_g = out_acc.cpu().numpy()
        t_g = out_tok.cpu().numpy()
        kv_gh = kv_g.cpu().numpy()
        ema_gh = ema_g.cpu().numpy().astype(np.float64)
        a_o = res["accept_len"]
        t_o = res["out_tokens"]
        k_eff = res["k_eff"]
        rep.rows += B * (K + 1)
        rep.rows_read += int((k_eff + 1).sum())
        rep.accepted += int(a_o.sum())
        rep.drafted += int(k_eff.sum())
        rep.count_accepts(a_o)
        rep.gated += int(((k.numpy() > 0) & (k_eff == 0)).sum())
        bad = compare(step, a_g, t_g, kv_gh, ema_gh, res, rep)
        if cooling:
            assert np.array_equal(cool_g.cpu().numpy(), res["gate_state"]), f"step {step}: cooling counts differ"
            cool_o = res["gate_state"]
        # ---- commit: both sides append their own tokens
        sp.spec_append(hist_g, lens_g, out_tok, out_acc)
        for b in range(B):
            a = int(a_o[b])
            hist_o[b, lens_o[b]:lens_o[b] + a + 1] = t_o[b, :a + 1]
            if stats is not None:
                on.extend_stats(stats[b], hist_o[b], int(lens_o[b]), int(lens_o[b]) + a + 1)
            lens_o[b] += a + 1
        kv_o = res["kv_len"]
        ema_o = res["ema"].astype(np.float32).astype(np.float64)
        if bad.any():  # overwrite the GPU state with the oracle's
            hist_g.copy_(torch.from_numpy(hist_o.astype(np.int32)))
            lens_g.copy_(torch.from_numpy(lens_o.astype(np.int32)))
            ema_g.copy_(torch.from_numpy(ema_o.astype(np.float32)))
        else:
            assert np.array_equal(lens_g.cpu().numpy(), lens_o)
            assert np.array_equal(hist_g.cpu().numpy(), hist_o)
            assert np.abs(ema_g.cpu().numpy().astype(np.float64) - ema_o).max(initial=0.0) <= EMA_TOL
        if use_ngram:
            if bad.any():  # the table is a function of the history: rebuild it
                table.reset()
            sp.ngram_update(table, hist_g, lens_g)
        rep.steps += 1
    status = sp.get_status(clear=True)
    assert status == 0, f"device status bits set: {sp.status_names(status)}"
    assert rep.excused <= EXCUSE_RATE * rep.rows, \
        f"{rep.excused} excused rows out of {rep.rows} exceed 1e-5:\n" + "\n".join(rep.notes)
    if table is not None:
        table.close()
    return rep
