#!/usr/bin/env python
"""Benchmark of the speculative-decoding hot path (n-gram draft -> verify ->
append -> n-gram update) on GB300, through the library's public API.

One step = one pass of the whole path over one batch: ngram_draft,
spec_verify, spec_append and ngram_update, with the target logits already
resident in HBM (a rotating set of synthetic batches larger than L2).
Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5]
    python bench.py --impl reference ...   # the fp64 oracle on the host cores
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_draft_ngram_gb300 import workloads as wl  # noqa: E402

METRIC = "spec_verify rows/s (B*(K+1) logit rows)"
UNIT = "rows/s"
DESCR = {
    "c2": "Qwen3-4B-shaped verify: B=1 V=151936 K=4 bf16 N(0,1)*4 logits, draft boosted to rowmax+6 w.p. 0.5, "
          "T=0.6, history 4096 Zipf(1.05) with 32-token copied spans, n-gram drafts",
    "c3": "Gemma-4-E2B-shaped continuous batch: B=64 V=262144 K=4 bf16 N(0,1)*8 logits, soft cap 30, T=1, "
          "histories U[512,8192] Zipf(1.1) with copied spans, n-gram drafts, EMA gate (tau 0.1, thr 0.5), "
          "boost w.p. U[0.2,0.9] per sequence",
    "c4": "dense-q verify: B=32 V=151936 K=4 T=0.6 bf16 N(0,1)*4 target, fp32 q = softmax((target+N(0,0.5))/0.6), "
          "drafts sampled from q, Leviathan accept + residual resampling",
    "c5": "large batch: B=256 V=151936 k_b~U{0..4} bf16 N(0,1)*4 logits, repetition penalty 1.1 over the last "
          "64 tokens, T=0.6, histories 32768 Zipf(1.05) with 64-token copied spans, n-gram update each step",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="c5", choices=sorted(DESCR))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the other workloads' verify timings")
    ap.add_argument("--schedule", default="split", choices=["split", "fused"],
                    help="spec_verify's kernel schedule in the timed loop (default: the library's default)")
    ap.add_argument("--early-exit", action="store_true", help="single-kernel schedule only: early exit")
    ap.add_argument("--cpu-sample", type=int, default=0, help="sequences in the oracle sample (0: auto)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (smaller profiler captures only)")
    ap.add_argument("--lmhead-batch", type=int, default=0,
                    help="only the fused LM head + verify measurement at this batch (profiler captures); prints its JSON")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_config(name: str, steps_total: int, rank: int, batch: int = 0) -> wl.Config:
    """The workload of one rank: same shapes on every rank, its own data and
    sampler seeds (weak scaling: each rank verifies an independent batch)."""
    cfg = wl.get(name)
    return wl.get(name, steps=max(cfg.steps, steps_total), data_seed=cfg.data_seed + 7919 * rank,
                  sampler_seed=cfg.sampler_seed + rank, B=batch or cfg.B)


def max_over_ranks(x: float, device) -> float:
    """Maximum of a per-rank value over all ranks (x itself on one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, bf16 copy)"
    return 6800.0, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def source_hash() -> str:
    h = hashlib.sha256()
    for f in ("verify.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_draft_ngram_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"verify_stream_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_launch_full")


class Clocks:
    """nvidia-smi sampler running during the timed region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = None
        self.ident = ident

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "20"]
            if self.ident:
                cmd += ["-i", self.ident]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        """Summary of the samples whose timestamps fall in window = (t0, t1)
        (host wall-clock seconds bracketing the timed region)."""
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if window is not None:
            from datetime import datetime
            keep = []
            for r in rows:
                try:
                    ts = datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if window[0] <= ts <= window[1]:
                    keep.append(r)
            rows = keep or rows[-1:]
        if not rows:
            return None
        num = lambda x: x.replace(".", "", 1).isdigit()  # noqa: E731
        sm = [float(r[2]) for r in rows if num(r[2])]
        mx = [float(r[3]) for r in rows if num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm

class Path:
    """Device state of one workload and its step function."""

    def __init__(self, name, steps_total, device, seed_offset=0, batch=0):
        import speculative_decoding_draft_ngram_gb300 as sp
        self.sp = sp
        cfg = rank_config(name, steps_total, seed_offset, batch)
        self.cfg = cfg
        self.dev = device
        B, K, V = cfg.B, cfg.K, cfg.V
        self.hist, self.lens = wl.histories(cfg, device)
        self.ngram = not cfg.dense
        if self.ngram:
            self.table = sp.NgramTable(B, V, B * cfg.hist_cap, device=device)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            sp.ngram_update(self.table, self.hist, self.lens)
            torch.cuda.synchronize()
            self.build_ms = (time.perf_counter() - t0) * 1e3
        g = wl._gen(cfg.data_seed + 1, device)
        set_bytes = B * (K + 1) * V * (2 if cfg.dtype == "bf16" else 4)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.n_sets = max(3, math.ceil(2 * l2 / set_bytes) + 1)
        self.set_bytes = set_bytes
        self.logits = [wl.step_logits(cfg, g, device=device) for _ in range(self.n_sets)]
        self.q = [None] * self.n_sets
        self.dsets = [None] * self.n_sets
        if cfg.dense:
            for i in range(self.n_sets):
                self.q[i], self.dsets[i] = wl.dense_draft(cfg, self.logits[i], g)
        self.limits = (wl.draft_limits(cfg, g, device) if not cfg.k_uniform else
                       torch.randint(0, K + 1, (steps_total, B), generator=g, device=device, dtype=torch.int32))
        self.bprob = wl.boost_probs(cfg, device)
        # the target-model stand-in's row maxima, per rotating batch (the boost restores the logits each step)
        self.rowmax = ([x[:, :K].amax(dim=-1).float() for x in self.logits] if cfg.boost is not None
                       else [None] * self.n_sets)
        zcdf = wl.zipf_cdf(cfg.zipf_ids or cfg.V, cfg.zipf_s, device)
        self.fallback = [wl.fallback_drafts(cfg, g, device, zcdf) for _ in range(16)] if cfg.topup else None
        self.kbuf = torch.zeros((steps_total, B), dtype=torch.int32, device=device)
        self.drafts = torch.full((B, K), -1, dtype=torch.int32, device=device)
        self.kfull = torch.full((B,), K, dtype=torch.int32, device=device)
        self.kv = self.lens.clone()
        self.ema = torch.ones(B, dtype=torch.float32, device=device)
        self.out = torch.empty((B, K + 1), dtype=torch.int32, device=device)
        self.acc = torch.empty((B,), dtype=torch.int32, device=device)
        self.ws = sp.spec_verify_workspace(B, K, V, device)
        self.params = sp.VerifyParams(temperature=cfg.temperature, softcap=cfg.softcap, rep_penalty=cfg.rep_penalty,
                                      rep_window=cfg.rep_window, gate_enabled=cfg.gate, seed=cfg.sampler_seed)
        # library kernels per step: spec_verify (the streaming kernel and the per-sequence decision
        # kernel, + the residual pass with dense q at T > 0), then spec_commit (append + index +
        # next drafts) or, without n-gram drafts, spec_append
        self.launches_per_step = (3 if cfg.dense and cfg.temperature > 0 else 2) + 1
        self.g = g

    def _limits(self, s):
        cfg = self.cfg
        lim = self.limits[s] if cfg.k_uniform else None
        fb = self.fallback[s % 16] if self.fallback is not None else None
        return lim, fb

    def first_drafts(self, s):
        """Drafts of step s from the table (the steps after it get theirs from spec_commit)."""
        if self.ngram:
            lim, fb = self._limits(s)
            self.sp.ngram_draft(self.table, self.hist, self.lens, self.cfg.K, k_limit=lim, out_drafts=self.drafts,
                                out_k=self.kbuf[s], fallback=fb)

    def step(self, s, logits, ev=None, rowmax=None):
        """One pass of the hot path: verify step s's drafts, then commit (append the
        emitted tokens, index them, draft step s + 1); ev = (start, end) events
        around spec_verify; rowmax: the row maxima of `logits` (boosted workloads)."""
        sp, cfg = self.sp, self.cfg
        if self.ngram:
            drafts, k, q = self.drafts, self.kbuf[s], None
        else:
            i = s % self.n_sets
            drafts, k, q = self.dsets[i], self.kfull, self.q[i]
        saved = None
        if cfg.boost is not None:
            # target-model stand-in (not the library's work): it agrees with a draft
            # w.p. rho_b; it runs before the step's library events
            saved = self._boost(logits, drafts, k, rowmax)
        self.params.step = s
        if ev is not None:
            ev[0].record()
        sp.spec_verify(logits, drafts, q, k, self.hist, self.lens, self.params, self.kv, self.ema, self.out,
                       self.acc, self.ws)
        if ev is not None:
            ev[1].record()
        if self.ngram:
            lim, fb = self._limits(s + 1)
            sp.spec_commit(self.table, self.hist, self.lens, self.out, self.acc, cfg.K, k_limit=lim, fallback=fb,
                           out_drafts=self.drafts, out_k=self.kbuf[s + 1])
        else:
            sp.spec_append(self.hist, self.lens, self.out, self.acc)
        if ev is not None:
            ev[2].record()
        if saved is not None:
            logits.view(-1)[saved[0]] = saved[1]

    def _boost(self, logits, drafts, k, rowmax=None):
        B, K1, V = logits.shape
        coin = torch.rand((B, K1 - 1), generator=self.g, device=logits.device) < self.bprob[:, None]
        j = torch.arange(K1 - 1, device=logits.device)[None, :]
        ok = coin & (j < k[:, None]) & (drafts >= 0)
        # every (b, j) slot is written (the old value where the coin says no), so no
        # data-dependent count ever reaches the host
        idx = ((torch.arange(B, device=logits.device)[:, None] * K1 + j) * V + drafts.clamp(min=0).long()).view(-1)
        if rowmax is None:
            rowmax = logits[:, :K1 - 1].amax(dim=-1)
        old = logits.view(-1)[idx].clone()
        newv = torch.where(ok.view(-1), (rowmax.float() + 6.0).to(logits.dtype).view(-1), old)
        logits.view(-1)[idx] = newv
        return idx, old

    def time_verify(self, calls: int = 60):
        """Device time of spec_verify alone: `calls` back-to-back calls on the
        workload's current state, each on the next logit batch of the rotation
        (the batches together are larger than L2, so every call reads its
        logits from HBM), bracketed by one pair of CUDA events on the
        launching stream.  A first, untimed pass of the same calls records the
        EMA before each call, so the rows each call reads (rows 0..k_eff of
        every sequence, with the gate) are known exactly; kv_len and the EMA
        are restored before the timed pass, which repeats the same calls.
        A second pass of the same calls times the streaming kernel alone (the
        library records a marker event right after it).  Returns (mean seconds
        per call, mean rows read per call, mean seconds of the streaming kernel)."""
        sp, cfg = self.sp, self.cfg
        kv0, ema0 = self.kv.clone(), self.ema.clone()
        s0 = self.n_sets * 1000
        drafts, k, q = (self.drafts, self.kbuf[s0 % self.kbuf.shape[0]], None) if self.ngram else (None, self.kfull, None)
        if self.ngram:
            self.first_drafts(s0 % self.kbuf.shape[0])

        def call(i):
            j = i % self.n_sets
            dr, qq = (drafts, q) if self.ngram else (self.dsets[j], self.q[j])
            self.params.step = s0 + i
            sp.spec_verify(self.logits[j], dr, qq, k, self.hist, self.lens, self.params, self.kv, self.ema,
                           self.out, self.acc, self.ws)

        n = calls + 3
        emas = []
        for i in range(n):
            emas.append(self.ema.clone())
            call(i)
        torch.cuda.synchronize()
        rows = []
        for i in range(3, n):
            keff = k
            if self.params.gate_enabled:
                keff = torch.where((k > 0) & ~(emas[i] >= self.params.ema_thresh), torch.zeros_like(k), k)
            rows.append(int((keff + 1).sum().item()))
        self.kv.copy_(kv0)
        self.ema.copy_(ema0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(3):
            call(i)
        e0.record()
        for i in range(3, n):
            call(i)
        e1.record()
        torch.cuda.synchronize()
        # the streaming kernel alone: the same calls again, an event before each call and
        # the library's marker event right after its streaming kernel
        self.kv.copy_(kv0)
        self.ema.copy_(ema0)
        spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
        for _, b in spans:
            b.record()  # the marker events must exist before the library records them
        for i in range(3):
            call(i)
        for i in range(3, n):
            spans[i - 3][0].record()
            sp.set_verify_marker(spans[i - 3][1])
            call(i)
        sp.set_verify_marker(None)
        torch.cuda.synchronize()
        k1_s = statistics.mean(a.elapsed_time(b) for a, b in spans) / 1e3
        self.kv.copy_(kv0)
        self.ema.copy_(ema0)
        return e0.elapsed_time(e1) / 1e3 / calls, statistics.mean(rows), k1_s

    def rows_read(self, steps):
        cfg = self.cfg
        if self.ngram:
            return int((self.kbuf[:steps] + 1).sum().item())
        return steps * cfg.B * (cfg.K + 1)


def verify_summary(path, peak, calls=60):
    """spec_verify alone on the workload's current state: the whole call and its
    streaming kernel against the HBM roofline (see Path.time_verify)."""
    cfg = path.cfg
    v_avg_s, v_rows, k1_s = path.time_verify(calls)
    elem = 2 if cfg.dtype == "bf16" else 4
    call_bytes = v_rows * cfg.V * elem + cfg.B * 4 * (2 * cfg.K + 8)
    k1_bytes = v_rows * cfg.V * elem
    return {
        "verify_us": v_avg_s * 1e6,
        "rows_read_per_call": v_rows,
        "rows_read_per_s": v_rows / v_avg_s,
        "nominal_rows_per_s": cfg.B * (cfg.K + 1) / v_avg_s,
        "verify_logits_gbs": call_bytes / v_avg_s / 1e9,
        "verify_call_frac": call_bytes / v_avg_s / 1e9 / peak,
        "stream_kernel_us": k1_s * 1e6,
        "stream_kernel_frac": k1_bytes / k1_s / 1e9 / peak,
    }


# Workloads measured beside the headline (spec_verify alone, same process):
# name -> (workload, what is timed, steps run first, gate forced open)
SUB_WORKLOADS = {
    "c5_fused": ("c5", "c5 under the single-kernel schedule (whole rows per CTA, each row decided by the CTA "
                       "that streamed it)", 8, dict(schedule=1)),
    "c5_early_exit": ("c5", "c5, single-kernel schedule with early exit: the rows past a known first rejection "
                            "are not read (same outputs)", 8, dict(schedule=1, early_exit=True)),
    "c3_gate_open": ("c3", "c3 with every sequence verifying its k drafts (gate forced open for the timing): the "
                           "soft-capped accept rows at V=262144", 8, dict(gate_enabled=False)),
    "c3_steady": ("c3", "c3 after 150 steps of the whole path with the EMA gate (tau 0.1, thr 0.5) as configured",
                  150, {}),
    "c4": ("c4", "c4 dense q: accept rows, decisions and the residual samples", 8, {}),
    "c2": ("c2", "c2 latency case (B=1), T=0.6", 8, {}),
}


def measure_sub_workloads(dev, peak, names):
    out = {}
    for name in names:
        wname, what, warm, overrides = SUB_WORKLOADS[name]
        path = Path(wname, warm + 2 * 70 + 16, dev)
        path.first_drafts(0)
        for s in range(warm):
            path.step(s, path.logits[s % path.n_sets], rowmax=path.rowmax[s % path.n_sets])
        torch.cuda.synchronize()
        for k_, v_ in overrides.items():
            setattr(path.params, k_, v_)
        d = {"what": what, "B": path.cfg.B, "V": path.cfg.V, "K": path.cfg.K}
        d.update(verify_summary(path, peak))
        out[name] = d
        del path
        torch.cuda.empty_cache()
    return out


def step_summary(acc, k, K):
    """Per-step metrics of the steps run after the timed loop: acc, k [steps, B]
    (accept lengths, drafts offered).  Each call emits a + 1 tokens per sequence."""
    a = acc.long()
    hist = torch.bincount(a.flatten(), minlength=K + 1)[:K + 1].tolist()
    offered = int(k.long().sum())
    return {
        "steps": int(a.shape[0]),
        "accept_len_hist": hist,                                   # counts of a = 0..K over steps x sequences
        "tokens_per_sequence_step": float((a + 1).double().mean()),
        "tokens_per_step": float((a + 1).double().sum(1).mean()),   # the whole batch
        "drafts_offered_per_step": float(k.long().sum(1).double().mean()),
        "acceptance_rate": (float(a.sum()) / offered) if offered else None,
    }


def measure_lmhead(dev, B=256, K=4, V=151936, d=2560, reps=20):
    """Fused LM head + verify (spec_verify_lmhead) at the c5 batch shape with a
    Qwen3-4B-sized head (d = 2560, V = 151936), no repetition penalty (the fused
    path does not take it), T = 0.6: the whole call, the LM-head kernel alone
    (an event after it), and for comparison the same logits from a cuBLAS
    matmul followed by spec_verify.  Inputs: random bf16 hidden states and
    weights (the weight, 778 MB, is larger than L2, so every call reads it
    from HBM)."""
    import speculative_decoding_draft_ngram_gb300 as sp
    g = torch.Generator(device=dev).manual_seed(21)
    hidden = torch.randn((B, K + 1, d), generator=g, device=dev).to(torch.bfloat16)
    weight = (torch.randn((V, d), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    drafts = torch.randint(0, V, (B, K), generator=g, device=dev, dtype=torch.int32)
    k = torch.randint(0, K + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    logits = torch.empty((B, K + 1, V), dtype=torch.bfloat16, device=dev)
    kv = torch.full((B,), 1000, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws_f = sp.spec_verify_lmhead_workspace(B, K, V, device=dev)
    ws_s = sp.spec_verify_workspace(B, K, V, device=dev)
    p = sp.VerifyParams(temperature=0.6, gate_enabled=False, seed=3, step=0)

    def fused():
        sp.spec_verify_lmhead(hidden, weight, logits, drafts, None, k, None, None, p, kv, ema, out, acc, ws_f)

    def unfused():
        torch.matmul(hidden.view(-1, d), weight.t(), out=logits.view(-1, V))
        sp.spec_verify(logits, drafts, None, k, None, None, p, kv, ema, out, acc, ws_s)

    def timed(fn, marker=False):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        m = torch.cuda.Event(enable_timing=True)
        m.record()
        if marker:
            sp.set_verify_marker(m)
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        first = []
        for i in range(reps):
            e0[i].record()
            fn()
            e1[i].record()
            if marker:
                torch.cuda.synchronize()
                first.append(e0[i].elapsed_time(m))
        torch.cuda.synchronize()
        if marker:
            sp.set_verify_marker(None)
        call = statistics.mean(e0[i].elapsed_time(e1[i]) for i in range(reps))
        return call, (statistics.mean(first) if first else None)

    call_f, head_f = timed(fused, marker=True)
    call_f2, _ = timed(fused)
    call_u, _ = timed(unfused)
    flops = 2.0 * B * (K + 1) * V * d
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        with open(pp) as f:
            peaks = json.load(f)
    peak_tf = float(peaks.get("bf16_tflops", 1900.0))
    st = sp.get_status(clear=True)
    res = {
        "what": "fused LM head (tcgen05 GEMM, bf16 logits and per-block records in its epilogue) + decision "
                "kernel, c5 batch shape, d=2560, no penalty, T=0.6",
        "B": B, "K": K, "V": V, "d": d,
        "call_us": call_f2 * 1e3,
        "lmhead_kernel_us": head_f * 1e3,
        "lmhead_tflops": flops / (head_f * 1e-3) / 1e12,
        "lmhead_frac_of_bf16_peak": flops / (head_f * 1e-3) / 1e12 / peak_tf,
        "peak_bf16_tflops": peak_tf,
        "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)" if peaks else "fallback 1.9 PF",
        "unfused_cublas_matmul_plus_spec_verify_us": call_u * 1e3,
        "status": sp.status_names(st),
    }
    del hidden, weight, logits, ws_f, ws_s
    torch.cuda.empty_cache()
    return res


def measure_graph_step(dev, name="c2", steps=200):
    """Whole-step CUDA-graph replay against the same step launched call by call:
    spec_verify (decode step read from a device counter) -> spec_commit ->
    KV block trim and reserve -> step counter advance, on fixed buffers (one
    logits batch, the drafts and counts written in place by spec_commit).
    Returns device microseconds per step for both, over `steps` steps."""
    import speculative_decoding_draft_ngram_gb300 as sp
    path = Path(name, 24, dev)
    cfg = path.cfg
    path.first_drafts(0)
    for s in range(8):
        path.step(s, path.logits[s % path.n_sets], rowmax=path.rowmax[s % path.n_sets])
    torch.cuda.synchronize()
    logits = path.logits[0]
    k = path.kbuf[8].clone() if path.ngram else path.kfull
    lim, fb = path._limits(9)
    pool = sp.KvPool(num_blocks=cfg.B * 4096, B=cfg.B, max_blocks=4096, block_size=16, device=dev)
    pool.reserve(path.kv, cfg.K + 1)
    step_t = torch.full((1,), 8, dtype=torch.int64, device=dev)
    params = dataclasses.replace(path.params, step_dev=step_t)

    def one():
        sp.spec_verify(logits, path.drafts, None, k, path.hist, path.lens, params, path.kv, path.ema, path.out,
                       path.acc, path.ws)
        if path.ngram:
            sp.spec_commit(path.table, path.hist, path.lens, path.out, path.acc, cfg.K, k_limit=lim, fallback=fb,
                           out_drafts=path.drafts, out_k=k)
        else:
            sp.spec_append(path.hist, path.lens, path.out, path.acc)
        pool.trim(path.kv)
        pool.reserve(path.kv, cfg.K + 1)
        sp.step_advance(step_t)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    for _ in range(3):
        one()
    eager_us = timed(one, steps)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        one()
    g.replay()
    graph_us = timed(g.replay, steps)
    st = sp.get_status(clear=True)
    del path
    torch.cuda.empty_cache()
    return {"what": f"{name}: one whole step (verify, commit, KV trim + reserve, step advance) per graph replay, "
                    "against the same calls launched one by one",
            "step_us_graph": graph_us, "step_us_eager": eager_us, "steps": steps,
            "status": sp.status_names(st)}


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import speculative_decoding_draft_ngram_gb300 as sp
    sp.load()
    total_steps = args.warmup + args.steps
    e2e_steps = 0 if args.no_e2e else min(args.steps, 200)
    path = Path(args.workload, 2 * total_steps + e2e_steps + 8, dev, seed_offset=rank, batch=args.batch)
    cfg = path.cfg
    if args.schedule == "fused":
        path.params.schedule = 1
        path.params.early_exit = bool(args.early_exit)
        path.launches_per_step = 2
    stream = torch.cuda.current_stream(dev)

    # ---- device-resident timed loop
    path.first_drafts(0)
    for s in range(args.warmup):
        path.step(s, path.logits[s % path.n_sets], rowmax=path.rowmax[s % path.n_sets])
    torch.cuda.synchronize()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(min(args.steps, 20))]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = Clocks(dev) if rank == 0 else None
    if clocks:
        clocks.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    base = args.warmup
    wall0 = time.time()
    torch.cuda.nvtx.range_push("timed")  # lets a profiler keep only the timed steps' launches
    t_start.record(stream)
    for i in range(args.steps):
        s = base + i
        path.step(s, path.logits[s % path.n_sets], rowmax=path.rowmax[s % path.n_sets])
    t_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall1 = time.time()
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop((wall0, wall1)) if clocks else None
    ms = t_start.elapsed_time(t_end)
    # rows of the timed steps only
    rows_read = path.rows_read(base + args.steps) - path.rows_read(base)
    # the split of a step (events between its calls; outside the timed loop, since an
    # event between two kernels stops the next one from launching early)
    nbreak = len(evs)
    acc_steps, k_steps = [], []   # per-step accept lengths and draft counts (outside the timed region)
    for i in range(nbreak):
        s = base + args.steps + i
        k_steps.append((path.kbuf[s] if path.ngram else path.kfull).clone())
        path.step(s, path.logits[s % path.n_sets], evs[i], rowmax=path.rowmax[s % path.n_sets])
        acc_steps.append(path.acc.clone())
    torch.cuda.synchronize()
    step_metrics = step_summary(torch.stack(acc_steps).cpu(), torch.stack(k_steps).cpu(), cfg.K)
    verify_ms = [a.elapsed_time(b) for a, b, _ in evs]
    library_ms = [a.elapsed_time(c) for a, _, c in evs]   # spec_verify + spec_commit / spec_append
    rows_nominal = args.steps * cfg.B * (cfg.K + 1)
    ms_max = max_over_ranks(ms, dev)
    status = sp.get_status(clear=True)

    # ---- end to end: host logits -> device, step, results -> host
    e2e = None
    if e2e_steps:
        host = [x.cpu().pin_memory() for x in path.logits[:3]]
        dbuf = torch.empty_like(path.logits[0])
        out_h = torch.empty(path.out.shape, dtype=torch.int32).pin_memory()
        acc_h = torch.empty(path.acc.shape, dtype=torch.int32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        base2 = base + args.steps + nbreak
        for i in range(3):  # warm the copy path
            dbuf.copy_(host[i % 3], non_blocking=True)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        e0.record(stream)
        for i in range(e2e_steps):
            dbuf.copy_(host[i % 3], non_blocking=True)
            path.step(base2 + i, dbuf, rowmax=path.rowmax[i % 3])
            out_h.copy_(path.out, non_blocking=True)
            acc_h.copy_(path.acc, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": ws * e2e_steps * cfg.B * (cfg.K + 1) / (ems / 1e3), "unit": UNIT,
               "bound": "the host-to-device copy of each step's whole logit batch [B, K+1, V] from pinned memory",
               "h2d_bytes_per_step": int(dbuf.numel() * dbuf.element_size()),
               "d2h_bytes_per_step": int(out_h.numel() * 4 + acc_h.numel() * 4), "steps": e2e_steps,
               "ms_per_step": ems / e2e_steps}
        status |= sp.get_status(clear=True)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_src = measured_peaks()
    # the kernels' own time (no launch gaps), for the roofline
    v_avg_s, v_rows, k1_s = path.time_verify()
    elem = 2 if cfg.dtype == "bf16" else 4
    per_launch_bytes = int(v_rows * cfg.V * elem + cfg.B * 4 * (2 * cfg.K + 8))
    achieved = per_launch_bytes / v_avg_s / 1e9            # the whole spec_verify call
    k1_bytes = int(v_rows * cfg.V * elem)                   # the streaming kernel reads each active row once
    k1_achieved = k1_bytes / k1_s / 1e9
    step_verify_us = statistics.mean(verify_ms) * 1e3
    del path.logits[:]
    torch.cuda.empty_cache()
    subs = measure_sub_workloads(dev, peak, [n for n in SUB_WORKLOADS
                                             if SUB_WORKLOADS[n][0] != args.workload or SUB_WORKLOADS[n][3]]
                                 if not args.no_sub else [])
    if not args.no_sub:
        subs["c2_graph"] = measure_graph_step(dev, "c2")
        subs["c5_lmhead"] = measure_lmhead(dev)
    traffic = ncu_traffic(args.workload)
    line = {
        "metric": METRIC,
        "value": ws * rows_nominal / (ms_max / 1e3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {DESCR[args.workload]}",
            "schedule": args.schedule + (" + early exit" if args.early_exit else ""),
            "B": cfg.B, "K": cfg.K, "V": cfg.V, "logits_dtype": cfg.dtype,
            "l2": f"inputs larger than L2: {path.n_sets} rotating logit batches of {path.set_bytes / 1e6:.0f} MB",
            "parallelism": f"dp{ws} (independent sequences per GPU)",
        },
        "rows_read_per_s": ws * rows_read / (ms_max / 1e3),
        "library_ms_per_step": statistics.mean(library_ms),
        "verify_us": v_avg_s * 1e6,
        "verify_us_in_step": step_verify_us,
        "verify_logits_gbs": achieved,
        "verify_call_frac": achieved / peak,
        "roofline": {
            "bound": "hbm", "achieved": k1_achieved, "peak": peak, "unit": "GB/s", "frac": k1_achieved / peak,
            "traffic": traffic,
            "kernel": "verify_stream_kernel, the dominant kernel of spec_verify (the decision kernel and, with "
                      "dense q, the residual pass follow it; the whole call is verify_us / verify_logits_gbs); "
                      "60 calls on rotating logit batches larger than L2 together, a CUDA event before each call "
                      "and the library's marker event right after the streaming kernel",
            "kernel_us": k1_s * 1e6,
            "rows_per_launch": v_rows,
            "peak_source": peak_src,
            "algorithmic_bytes_per_launch": k1_bytes,
        },
        "gpu_launches": path.launches_per_step * args.steps,
        "e2e": e2e,
        "step_metrics": step_metrics,
        "workloads": subs,
        "clocks": clk,
        "device_status": sp.status_names(status),
    }
    if path.ngram:
        line["ngram_build_ms"] = path.build_ms
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- oracle arm

class OracleState:
    """A bounded sample of the workload's sequences, stepped by the oracle
    (worker w draws its own independent sequences: data seed + 7919 w)."""

    def __init__(self, name, nseq, worker=0):
        cfg = wl.get(name)
        cfg = wl.get(name, B=nseq, steps=max(cfg.steps, 64), data_seed=cfg.data_seed + 7919 * worker)
        self.cfg = cfg
        hist, lens = wl.histories(cfg, "cpu")
        self.hist = hist.numpy().astype(np.int64)
        self.lens = lens.numpy().astype(np.int64)
        self.g = wl._gen(cfg.data_seed + 1, "cpu")
        self.ema = np.ones(cfg.B)
        self.kv = self.lens.copy()

    def step(self, s):
        from oracle import ngram as on
        from oracle import verify as ov
        cfg = self.cfg
        logits = wl.step_logits(cfg, self.g)
        lim = wl.draft_limits(cfg, self.g).numpy()
        fb = wl.fallback_drafts(cfg, self.g)
        if cfg.dense:
            q, d = wl.dense_draft(cfg, logits, self.g)
            q, d, k = q.numpy(), d.numpy().astype(np.int64), np.full(cfg.B, cfg.K)
        else:
            d, k = on.draft_batch(self.hist, self.lens, cfg.K, k_limit=lim,
                                  fallback=None if fb is None else fb.numpy())
            q = None
        if cfg.boost is not None:
            logits = wl.apply_boost(cfg, logits, torch.from_numpy(d), torch.from_numpy(k),
                                    wl.boost_probs(cfg), self.g)
        p = ov.VerifyParams(temperature=cfg.temperature, softcap=cfg.softcap, rep_penalty=cfg.rep_penalty,
                            rep_window=cfg.rep_window, gate_enabled=cfg.gate, seed=cfg.sampler_seed, step=s)
        res = ov.spec_verify(logits.float().numpy(), d, q, k, self.hist, self.lens, p, self.kv,
                             self.ema.astype(np.float32))
        for b in range(cfg.B):
            a = int(res["accept_len"][b])
            self.hist[b, self.lens[b]:self.lens[b] + a + 1] = res["out_tokens"][b, :a + 1]
            self.lens[b] += a + 1
        self.kv = res["kv_len"]
        self.ema = res["ema"]
        return cfg.B * (cfg.K + 1)


AUTO_SAMPLE = {"c2": 1, "c3": 2, "c4": 3, "c5": 4}   # sequences per worker


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_worker_init():
    # one numpy thread per worker: the pool spreads the sequences over the cores
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    torch.set_num_threads(1)


def _oracle_worker(task):
    """One worker's share: its own independent sequences of the workload (its
    own data seed), stepped by the oracle; returns (rows, seconds)."""
    name, nseq, steps, worker, warm = task
    st = OracleState(name, nseq, worker)
    for s in range(warm):
        st.step(s)
    t0 = time.perf_counter()
    rows = sum(st.step(warm + s) for s in range(steps))
    return rows, time.perf_counter() - t0


def oracle_parallel(name, nseq_per_worker, steps, warm=0, workers=None):
    """The oracle, as it stands, on all host cores: one process per core (spawned,
    so no CUDA state is inherited), each stepping its own sequences.  Returns
    (rows/s over the parallel region, workers, rows, wall seconds)."""
    import multiprocessing as mp
    workers = workers or (os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_oracle_worker_init) as pool:
        pool.map(_noop, range(workers))          # workers up and their imports done
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(name, nseq_per_worker, steps, w, warm) for w in range(workers)])
        wall = time.perf_counter() - t0
    rows = sum(r for r, _ in res)
    return rows / wall, workers, rows, wall


def _noop(_):
    return 0


def cpu_baseline(name, nseq=0, steps=4):
    """Time the oracle, as it stands, on a bounded sample of the workload, on every host core."""
    nseq = nseq or AUTO_SAMPLE[name]
    v, workers, rows, wall = oracle_parallel(name, nseq, steps)
    return {"value": v, "unit": UNIT, "cores": workers, "kind": "oracle", "cpu_model": cpu_model(),
            "nproc": os.cpu_count(),
            "sample": f"{workers} worker processes (one per host core, one numpy thread each), each stepping "
                      f"{nseq} independent sequences of workload {name} for {steps} full steps (n-gram draft "
                      f"from the history, fp64 verify, append); {rows} nominal rows in {wall:.1f} s wall"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    nseq = args.cpu_sample or 1   # sequences per worker per step: keeps the run within minutes
    v, workers, rows, wall = oracle_parallel(args.workload, nseq, args.steps, warm=args.warmup)
    sample = (f"each step: {workers} worker processes (one per host core) x {nseq} sequence(s) of workload "
              f"{args.workload} (n-gram draft, fp64 verify, append); {args.steps} timed steps after "
              f"{args.warmup} warm-up steps; {rows} nominal rows in {wall:.1f} s wall")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCR[args.workload]}", "sampled_sequences": nseq * workers},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": workers, "kind": "oracle", "cpu_model": cpu_model(),
                         "nproc": os.cpu_count(), "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.lmhead_batch > 0:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_lmhead(dev, B=args.lmhead_batch)))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
