"""GPU parity of the whole hot path (draft -> verify -> append -> update)
against the fp64 oracle, in lockstep, on every workload at sizes the oracle
finishes in seconds.  V = 40000 spans two 64 KB chunks of the streaming
pass in bf16 (three in fp32) with a ragged tail, and 157 noise blocks;
V = 40001 takes the unaligned (scalar-load) path."""
import pytest

import speculative_decoding_draft_ngram_gb300 as sp
from speculative_decoding_draft_ngram_gb300 import workloads as wl

import lockstep

pytestmark = pytest.mark.gpu

V_SMALL = 40000

CASES = {
    "c1": (wl.get("c1"), 64, None),
    "c2_greedy": (wl.get("c2", V=V_SMALL, hist_len=(512, 512), steps=16), 16, 0.0),
    "c2_t06": (wl.get("c2", V=V_SMALL, hist_len=(512, 512), steps=16), 16, 0.6),
    "c2_literal_boost": (wl.get("c2", V=V_SMALL, hist_len=(512, 512), boost="literal", steps=8), 8, 0.6),
    "c3_softcap_gate": (wl.get("c3", B=6, V=V_SMALL, hist_len=(64, 700), steps=16), 16, None),
    "c3_f32": (wl.get("c3", B=4, V=V_SMALL, hist_len=(64, 700), dtype="f32", steps=8), 8, None),
    "c3_greedy_softcap": (wl.get("c3", B=4, V=V_SMALL, hist_len=(64, 700), steps=8), 8, 0.0),
    "c4_dense": (wl.get("c4", B=6, V=V_SMALL, steps=10), 10, None),
    "c4_dense_f32": (wl.get("c4", B=3, V=V_SMALL, dtype="f32", steps=6), 6, None),
    "c4_dense_greedy": (wl.get("c4", B=6, V=V_SMALL, steps=8), 8, 0.0),
    "c4_dense_greedy_f32": (wl.get("c4", B=3, V=V_SMALL, dtype="f32", steps=5), 5, 0.0),
    "c4_dense_softcap_penalty": (wl.get("c4", B=3, V=V_SMALL, softcap=20.0, rep_penalty=1.3,
                                        rep_window=32, steps=6), 6, None),
    "c5_penalty": (wl.get("c5", B=7, V=V_SMALL, hist_len=(1500, 1500), steps=10), 10, None),
    "c5_f32": (wl.get("c5", B=5, V=V_SMALL, hist_len=(1500, 1500), dtype="f32", steps=6), 6, None),
    "c5_greedy_penalty": (wl.get("c5", B=5, V=V_SMALL, hist_len=(1500, 1500), steps=6), 6, 0.0),
    "c5_penalty_below_one": (wl.get("c5", B=4, V=V_SMALL, hist_len=(1500, 1500), rep_penalty=0.8,
                                    steps=6), 6, None),
    "unaligned_v": (wl.get("c5", B=4, V=V_SMALL + 1, hist_len=(1500, 1500), steps=6), 6, None),
    "unaligned_v_dense": (wl.get("c4", B=3, V=V_SMALL + 3, steps=5), 5, None),
    "tiny_v": (wl.get("c1", V=5, zipf_ids=5, steps=24), 24, None),
    "k2_many_seqs": (wl.get("c5", B=33, K=2, V=3000, hist_len=(300, 300), steps=8), 8, None),
    "k0_bonus_only": (wl.get("c5", B=4, K=0, V=V_SMALL, hist_len=(300, 300), steps=5), 5, None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_lockstep(name):
    cfg, steps, T = CASES[name]
    rep = lockstep.run(cfg, steps, T=T)
    assert rep.steps == steps
    assert rep.excused == 0, rep.notes
    if cfg.K > 0:
        assert rep.drafted > 0
    if name in ("c2_t06", "c2_greedy", "c3_softcap_gate", "c1"):
        assert rep.accepted > 0
    # per-step metrics: one accept length per sequence and step, a + 1 tokens each
    n = sum(rep.accept_hist)
    assert n == rep.rows // (cfg.K + 1)
    assert sum(i * c for i, c in enumerate(rep.accept_hist)) == rep.accepted
    assert abs(rep.tokens_per_sequence_step() - (1 + rep.accepted / n)) < 1e-12


# A low starting EMA with the gate off: the EMA update runs from a state far
# from its fixed point (and, on the boosted workloads c2 and c3, climbs back
# during the run), and must still match the oracle's step by step.
LOW_EMA = {
    "c5_low_ema": (wl.get("c5", B=7, V=V_SMALL, hist_len=(1500, 1500), steps=10), 10, None),
    "c5_low_ema_penalty_below_one": (wl.get("c5", B=4, V=V_SMALL, hist_len=(1500, 1500), rep_penalty=0.8, steps=6),
                                     6, None),
    "c2_low_ema_boost": (wl.get("c2", V=V_SMALL, hist_len=(512, 512), steps=16), 16, 0.6),
    "c3_low_ema_softcap": (wl.get("c3", B=6, V=V_SMALL, hist_len=(64, 700), gate=False, steps=12), 12, None),
}


@pytest.mark.parametrize("name", list(LOW_EMA))
def test_lockstep_low_starting_ema(name):
    cfg, steps, T = LOW_EMA[name]
    rep = lockstep.run(cfg, steps, T=T, ema0=0.1)
    assert rep.steps == steps
    assert rep.excused == 0, rep.notes
    assert rep.drafted > 0
    if name.startswith(("c2", "c3")):
        assert rep.accepted > 0


def test_gate_turns_sequences_off():
    cfg = wl.get("c3", B=8, V=8000, hist_len=(64, 400), boost_prob=(0.0, 0.3), steps=20)
    rep = lockstep.run(cfg, 20)
    assert rep.gated > 0


def test_long_c1_run():
    # the tiny workload for its full 64 steps with three sampler seeds
    for seed in (8, 123, 99991):
        lockstep.run(wl.get("c1"), 64, seed=seed)


FULL = {
    # the benchmark's workloads at full size and launch configuration; the
    # oracle checks sampled sequences one by one
    "c5_full": (wl.get("c5"), 10, 8),
    "c3_full": (wl.get("c3"), 10, 6),
    "c4_full": (wl.get("c4"), 4, 4),
    "c4_full_greedy": (wl.get("c4"), 3, 3),
    "c2_full_greedy": (wl.get("c2"), 3, 1),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(name):
    cfg, steps, sample = FULL[name]
    T = 0.0 if name.endswith("greedy") else None
    rep = lockstep.run_sampled(cfg, steps, sample, T=T)
    assert rep.steps == steps and rep.excused == 0, rep.notes
    assert rep.drafted > 0


# The same cases under the other kernel schedule and with early exit: the
# outputs must not depend on either (the two-kernel schedule is the default;
# the single kernel; the single kernel skipping the rows past a known first
# rejection).
SCHEDULES = {
    "fused": dict(schedule=sp.capi.SCHEDULE_FUSED),
    "early_exit": dict(schedule=sp.capi.SCHEDULE_FUSED, early_exit=True),
}
SCHED_CASES = ["c1", "c2_greedy", "c2_t06", "c3_softcap_gate", "c3_greedy_softcap", "c4_dense", "c4_dense_greedy",
               "c5_penalty", "c5_f32", "c5_penalty_below_one", "unaligned_v", "tiny_v", "k2_many_seqs",
               "k0_bonus_only"]


@pytest.mark.parametrize("sched", list(SCHEDULES))
@pytest.mark.parametrize("name", SCHED_CASES)
def test_lockstep_schedules(name, sched):
    cfg, steps, T = CASES[name]
    rep = lockstep.run(cfg, steps, T=T, **SCHEDULES[sched])
    assert rep.steps == steps and rep.excused == 0, rep.notes


def test_lockstep_large_batch():
    # B = 2100 sequences (dense drafts: an n-gram table holds at most 512 sequences)
    cfg = wl.get("c4", B=2100, K=2, V=1000, steps=3)
    rep = lockstep.run(cfg, 3, oracle_chunk=256)
    assert rep.steps == 3 and rep.excused == 0


def test_single_kernel_schedule_rejects_large_batches():
    import torch
    B, K, V = 2049, 1, 64
    dev = "cuda"
    p = sp.VerifyParams(temperature=1.0, gate_enabled=False, schedule=sp.capi.SCHEDULE_FUSED)
    args = (torch.zeros((B, K + 1, V), device=dev), torch.zeros((B, K), dtype=torch.int32, device=dev), None,
            torch.zeros(B, dtype=torch.int32, device=dev), None, None, p, torch.zeros(B, dtype=torch.int32, device=dev),
            torch.ones(B, device=dev), torch.empty((B, K + 1), dtype=torch.int32, device=dev),
            torch.empty(B, dtype=torch.int32, device=dev), sp.spec_verify_workspace(B, K, V))
    with pytest.raises(sp.SpecngError, match="B <= 2048"):
        sp.spec_verify(*args)


@pytest.mark.parametrize("name", ["c5_full", "c3_full", "c4_full"])
def test_full_size_sampled_early_exit(name):
    cfg, steps, sample = FULL[name]
    rep = lockstep.run_sampled(cfg, min(steps, 4), sample, early_exit=True, schedule=sp.capi.SCHEDULE_FUSED)
    assert rep.excused == 0, rep.notes


# Gate variants (re-probe, cooling after a partial acceptance) and drafts on
# repeated n-gram evidence, on both schedules: GPU against the oracle, the
# cooling counts bit-exact every step.
VARIANTS = {
    "c3_probe_cool": (wl.get("c3", B=6, V=V_SMALL, hist_len=(64, 700), steps=30), 30, None,
                      dict(probe_interval=4, cool_steps=2)),
    "c3_probe_low_rho": (wl.get("c3", B=8, V=8000, hist_len=(64, 400), boost_prob=(0.0, 0.3), steps=30), 30, None,
                         dict(probe_interval=3)),
    "c5_cool": (wl.get("c5", B=7, V=V_SMALL, hist_len=(1500, 1500), steps=12), 12, None, dict(cool_steps=3)),
    "c2_cool_greedy": (wl.get("c2", V=V_SMALL, hist_len=(512, 512), steps=16), 16, 0.0, dict(cool_steps=1)),
    "c1_min_count": (wl.get("c1"), 40, None, dict(min_count=2)),
    "c5_min_count": (wl.get("c5", B=7, V=V_SMALL, hist_len=(1500, 1500), steps=8), 8, None, dict(min_count=2)),
}


@pytest.mark.parametrize("sched", ["split", "fused"])
@pytest.mark.parametrize("name", list(VARIANTS))
def test_lockstep_gate_variants(name, sched):
    cfg, steps, T, var = VARIANTS[name]
    extra = {} if sched == "split" else dict(schedule=sp.capi.SCHEDULE_FUSED)
    rep = lockstep.run(cfg, steps, T=T, **var, **extra)
    assert rep.steps == steps and rep.excused == 0, rep.notes
    if "probe_interval" in var:
        assert rep.gated > 0
