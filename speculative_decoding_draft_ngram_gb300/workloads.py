"""Seeded synthetic workloads for the verify / n-gram path.

Input synthesis only -- no step of the method is computed here.  The tests
feed the same arrays to the GPU library and to the oracle; the benchmark
uses the same recipes.  Each config below is one synthetic workload of the
verify path; where a recipe leaves a detail open (the boosts, the copied
spans, the draft top-up), the choice is stated beside it.

  c1  tiny: B=1, V=32, K=4, fp32 logits N(0,1)*3 fresh per step, T=1, no soft
      cap; history of 256 Zipf(1.1) tokens over 32 ids with one fixed 8-token
      span placed at every 32-token boundary; n-gram drafts, EMA gate on.
  c2  Qwen3-4B-shaped: B=1, V=151936, K=4, bf16 N(0,1)*4; a draft's logit is
      boosted w.p. 0.5 ("intent": set to rowmax + 6, "literal": + 6); history
      4096 Zipf(1.05) tokens with 32-token copied spans; T = 0 and T = 0.6.
  c3  Gemma-4-E2B-shaped batch: B=64, V=262144, K=4, bf16 N(0,1)*8, soft cap
      30, T=1; histories of U[512, 8192] Zipf(1.1) tokens with 32-token copied
      spans; n-gram drafts, gate on; boost w.p. rho_b ~ U[0.2, 0.9] per
      sequence (rowmax + 6).
  c4  dense-q verify: B=32, V=151936, K=4, T=0.6, bf16 N(0,1)*4 target,
      q = softmax((target + N(0, 0.5)) / 0.6) in fp32, drafts d_i ~ q_{i-1}.
  c5  large batch: B=256, V=151936, k_b ~ U{0..4}, bf16 N(0,1)*4,
      repetition penalty 1.1 over the last 64 tokens, T=0.6; histories of
      32768 Zipf(1.05) tokens with 64-token copied spans; n-gram drafts
      capped at k_b.
  c2, c3 and c5 pad the n-gram drafts with Zipf proposals up to the
  per-sequence length (K, or k_b for c5) when the tables run dry.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    V: int
    K: int
    dtype: str                 # "bf16" or "f32"
    temperature: float
    softcap: float = 0.0
    rep_penalty: float = 1.0
    rep_window: int = 0
    gate: bool = False
    dense: bool = False
    steps: int = 100
    hist_len: Tuple[int, int] = (256, 256)
    zipf_s: float = 1.1
    zipf_ids: Optional[int] = None   # ids drawn from [0, zipf_ids) (default V)
    span: int = 32
    span_mode: str = "copy"           # "copy": copy an earlier window w.p. 0.5; "fixed"
    logit_scale: float = 4.0
    boost: Optional[str] = None       # None, "intent", "literal"
    boost_prob: Tuple[float, float] = (0.5, 0.5)   # per-sequence prob ~ U[lo, hi]
    k_uniform: bool = False           # k_b ~ U{0..K} per sequence per step
    topup: bool = False               # pad n-gram drafts with Zipf proposals up to the cap
    q_noise: float = 0.5
    data_seed: int = 0
    sampler_seed: int = 0

    @property
    def hist_cap(self) -> int:
        return self.hist_len[1] + self.steps * (self.K + 1) + 8

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


CONFIGS = {
    "c1": Config("c1", B=1, V=32, K=4, dtype="f32", temperature=1.0, gate=True, steps=64,
                 hist_len=(256, 256), zipf_s=1.1, span=8, span_mode="fixed", logit_scale=3.0,
                 data_seed=1001, sampler_seed=8),
    "c2": Config("c2", B=1, V=151936, K=4, dtype="bf16", temperature=0.6, gate=False, steps=1000,
                 hist_len=(4096, 4096), zipf_s=1.05, span=32, logit_scale=4.0, boost="intent",
                 topup=True, data_seed=1002, sampler_seed=9),
    "c3": Config("c3", B=64, V=262144, K=4, dtype="bf16", temperature=1.0, softcap=30.0, gate=True,
                 steps=500, hist_len=(512, 8192), zipf_s=1.1, span=32, logit_scale=8.0, boost="intent",
                 boost_prob=(0.2, 0.9), topup=True, data_seed=1003, sampler_seed=10),
    "c4": Config("c4", B=32, V=151936, K=4, dtype="bf16", temperature=0.6, dense=True, gate=False,
                 steps=500, hist_len=(1024, 1024), zipf_s=1.05, logit_scale=4.0, data_seed=1004,
                 sampler_seed=11),
    "c5": Config("c5", B=256, V=151936, K=4, dtype="bf16", temperature=0.6, rep_penalty=1.1,
                 rep_window=64, gate=False, steps=200, hist_len=(32768, 32768), zipf_s=1.05, span=64,
                 logit_scale=4.0, k_uniform=True, topup=True, data_seed=1005, sampler_seed=12),
}


def get(name: str, **overrides) -> Config:
    return replace(CONFIGS[name], **overrides)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_cdf(n_ids: int, s: float, device="cpu") -> torch.Tensor:
    """Cumulative law of a finite Zipf: P(rank r) ~ r^-s, r = 1..n_ids (id = r - 1)."""
    r = torch.arange(1, n_ids + 1, dtype=torch.float64, device=device)
    w = r.pow(-s)
    return torch.cumsum(w, 0) / w.sum()


def zipf_tokens(g: torch.Generator, shape, cdf: torch.Tensor) -> torch.Tensor:
    u = torch.rand(shape, generator=g, device=cdf.device, dtype=torch.float64)
    return torch.searchsorted(cdf, u).clamp_(max=cdf.numel() - 1).to(torch.int32)


def histories(cfg: Config, device="cpu", seed: Optional[int] = None):
    """(history [B, hist_cap] int32, lens [B] int32) following cfg's recipe."""
    g = _gen(cfg.data_seed if seed is None else seed, device)
    n_ids = cfg.zipf_ids or cfg.V
    cdf = zipf_cdf(n_ids, cfg.zipf_s, device)
    lo, hi = cfg.hist_len
    L = hi
    if lo == hi:
        lens = torch.full((cfg.B,), hi, dtype=torch.int32, device=device)
    else:
        lens = torch.randint(lo, hi + 1, (cfg.B,), generator=g, device=device, dtype=torch.int32)
    hist = torch.full((cfg.B, cfg.hist_cap), -1, dtype=torch.int32, device=device)
    tok = zipf_tokens(g, (cfg.B, L), cdf)
    span = cfg.span
    if cfg.span_mode == "fixed":
        fixed = zipf_tokens(g, (cfg.B, span), cdf)
        for s0 in range(0, L - span + 1, 32):
            tok[:, s0:s0 + span] = fixed
    else:
        rows = torch.arange(cfg.B, device=device)[:, None]
        off = torch.arange(span, device=device)[None, :]
        for s0 in range(span, L - span + 1, span):
            copy = torch.rand((cfg.B,), generator=g, device=device) < 0.5
            src = torch.randint(0, s0 - span + 1, (cfg.B,), generator=g, device=device)
            window = tok[rows, src[:, None] + off]
            tok[:, s0:s0 + span] = torch.where(copy[:, None], window, tok[:, s0:s0 + span])
    hist[:, :L] = tok
    pos = torch.arange(cfg.hist_cap, device=device)[None, :]
    hist = torch.where(pos < lens[:, None].long(), hist, torch.full_like(hist, -1))
    return hist, lens


def step_logits(cfg: Config, g: torch.Generator, B: Optional[int] = None, device="cpu") -> torch.Tensor:
    """Target logits [B, K+1, V]: N(0, 1) * scale, rounded to cfg.dtype (RNE for bf16)."""
    B = cfg.B if B is None else B
    x = torch.randn((B, cfg.K + 1, cfg.V), generator=g, device=device, dtype=torch.float32)
    return (x * cfg.logit_scale).to(cfg.torch_dtype)


def boost_probs(cfg: Config, device="cpu") -> torch.Tensor:
    g = _gen(cfg.data_seed + 17, device)
    lo, hi = cfg.boost_prob
    return lo + (hi - lo) * torch.rand((cfg.B,), generator=g, device=device, dtype=torch.float64)


def apply_boost(cfg: Config, logits: torch.Tensor, drafts: torch.Tensor, k: torch.Tensor,
                probs: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Stand-in for a target model that often agrees with the drafts: in row j,
    w.p. probs[b] the logit of d_{j+1} is set to rowmax + 6 ("intent") or
    raised by 6 ("literal").  Returns a new tensor."""
    if cfg.boost is None:
        return logits
    B, K1, V = logits.shape
    out = logits.clone()
    coin = torch.rand((B, K1 - 1), generator=g, device=logits.device, dtype=torch.float64) < probs[:, None]
    j = torch.arange(K1 - 1, device=logits.device)[None, :]
    valid = coin & (j < k[:, None].long()) & (drafts >= 0) & (drafts < V)
    bb, jj = torch.nonzero(valid, as_tuple=True)
    if bb.numel() == 0:
        return out
    d = drafts[bb, jj].long()
    if cfg.boost == "intent":
        newv = out[bb, jj].float().amax(dim=-1) + 6.0
    else:
        newv = out[bb, jj, d].float() + 6.0
    out[bb, jj, d] = newv.to(out.dtype)
    return out


def dense_draft(cfg: Config, logits: torch.Tensor, g: torch.Generator):
    """Draft-model stand-in: q = softmax((target + N(0, q_noise)) / T) in fp32,
    drafts d_{i+1} ~ q_i.  Returns (q [B, K, V] fp32, drafts [B, K] int32)."""
    B, K1, V = logits.shape
    tgt = logits[:, :K1 - 1].float()
    noise = torch.randn(tgt.shape, generator=g, device=logits.device, dtype=torch.float32) * cfg.q_noise
    q = torch.softmax((tgt + noise) / cfg.temperature, dim=-1)
    u = torch.rand((B, K1 - 1, 1), generator=g, device=logits.device, dtype=torch.float32)
    cdf = torch.cumsum(q, dim=-1)
    d = torch.searchsorted(cdf, u * cdf[..., -1:]).clamp_(max=V - 1).squeeze(-1).to(torch.int32)
    return q.contiguous(), d.contiguous()


def fallback_drafts(cfg: Config, g: torch.Generator, device="cpu", cdf: Optional[torch.Tensor] = None):
    """Stand-in for a second drafter: Zipf proposals [B, K] that pad the n-gram
    drafts up to the per-sequence length (None when cfg.topup is off)."""
    if not cfg.topup:
        return None
    if cdf is None:
        cdf = zipf_cdf(cfg.zipf_ids or cfg.V, cfg.zipf_s, device)
    return zipf_tokens(g, (cfg.B, cfg.K), cdf)


def draft_limits(cfg: Config, g: torch.Generator, device="cpu") -> torch.Tensor:
    """Per-sequence draft length caps: U{0..K} (c5) or K."""
    if cfg.k_uniform:
        return torch.randint(0, cfg.K + 1, (cfg.B,), generator=g, device=device, dtype=torch.int32)
    return torch.full((cfg.B,), cfg.K, dtype=torch.int32, device=device)
