"""CPU checks of the seeded input recipes: every config has the stated shapes,
scalars and value distributions (the synthetic stand-ins for the task's
workloads), and the generators are deterministic in their seeds."""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_ngram_gb300 import workloads as wl

# the workloads as stated: (B, V, K, logits dtype, T, soft cap, penalty, window, gate, dense, logit scale)
STATED = {
    "c1": (1, 32, 4, "f32", 1.0, 0.0, 1.0, 0, True, False, 3.0),
    "c2": (1, 151936, 4, "bf16", 0.6, 0.0, 1.0, 0, False, False, 4.0),
    "c3": (64, 262144, 4, "bf16", 1.0, 30.0, 1.0, 0, True, False, 8.0),
    "c4": (32, 151936, 4, "bf16", 0.6, 0.0, 1.0, 0, False, True, 4.0),
    "c5": (256, 151936, 4, "bf16", 0.6, 0.0, 1.1, 64, False, False, 4.0),
}


@pytest.mark.parametrize("name", list(STATED))
def test_configs_match_the_stated_workloads(name):
    c = wl.get(name)
    B, V, K, dt, T, cap, rep, win, gate, dense, scale = STATED[name]
    assert (c.B, c.V, c.K, c.dtype, c.temperature, c.softcap, c.rep_penalty, c.rep_window) == \
        (B, V, K, dt, T, cap, rep, win)
    assert (c.gate, c.dense, c.logit_scale) == (gate, dense, scale)


def test_seeds_follow_the_config_numbers():
    for i, name in enumerate(["c1", "c2", "c3", "c4", "c5"], start=1):
        c = wl.get(name)
        assert c.data_seed == 1000 + i and c.sampler_seed == 7 + i


def test_logits_scale_dtype_and_rounding():
    cfg = wl.get("c3", B=2, V=50000)
    x = wl.step_logits(cfg, wl._gen(5, "cpu"))
    assert x.shape == (2, cfg.K + 1, 50000) and x.dtype == torch.bfloat16
    xf = x.float()
    assert abs(xf.std().item() - 8.0) < 0.1 and abs(xf.mean().item()) < 0.05
    # bf16 values are the round-to-nearest-even images of the fp32 draws
    ref = (torch.randn((2, cfg.K + 1, 50000), generator=wl._gen(5, "cpu")) * 8.0).to(torch.bfloat16)
    assert torch.equal(x, ref)
    f32 = wl.step_logits(wl.get("c1"), wl._gen(1, "cpu"))
    assert f32.dtype == torch.float32 and f32.shape == (1, 5, 32)


def test_zipf_law():
    cdf = wl.zipf_cdf(1000, 1.1)
    t = wl.zipf_tokens(wl._gen(3, "cpu"), (400000,), cdf).numpy()
    assert t.min() >= 0 and t.max() < 1000
    counts = np.bincount(t, minlength=1000)
    # P(rank r) ~ r^-s: the frequencies of ids 0, 1, 3 (ranks 1, 2, 4) fall as 2^-1.1 per doubling
    assert abs(counts[0] / counts[1] - 2 ** 1.1) < 0.05
    assert abs(counts[1] / counts[3] - 2 ** 1.1) < 0.08


def test_histories_lengths_padding_and_copied_spans():
    cfg = wl.get("c3", B=16, V=5000, hist_len=(512, 2048))
    hist, lens = wl.histories(cfg)
    lens = lens.numpy()
    h = hist.numpy()
    assert lens.min() >= 512 and lens.max() <= 2048
    assert h.shape == (16, cfg.hist_cap)
    for b in range(16):
        assert (h[b, :lens[b]] >= 0).all() and (h[b, lens[b]:] == -1).all()
    # about half of the 32-token blocks after the first repeat an earlier window
    rep = tot = 0
    for b in range(16):
        row = h[b, :lens[b]]
        for s0 in range(32, lens[b] - 31, 32):
            blk = row[s0:s0 + 32]
            tot += 1
            win = np.lib.stride_tricks.sliding_window_view(row[:s0], 32)
            rep += bool((win == blk).all(axis=1).any())
    assert 0.4 < rep / tot < 0.6


def test_tiny_history_repeats_one_fixed_span():
    cfg = wl.get("c1")
    hist, lens = wl.histories(cfg)
    row = hist.numpy()[0, :int(lens[0])]
    assert row.max() < 32
    spans = [tuple(row[s0:s0 + 8]) for s0 in range(0, 256 - 7, 32)]
    assert len(set(spans)) == 1


def test_boost_probabilities_and_intent_boost():
    cfg = wl.get("c3", B=200, V=3000)
    p = wl.boost_probs(cfg).numpy()
    assert p.min() >= 0.2 and p.max() <= 0.9 and 0.45 < p.mean() < 0.65
    g = wl._gen(9, "cpu")
    cfg = wl.get("c2", B=64, V=3000)
    logits = wl.step_logits(cfg, g)
    drafts = torch.randint(0, 3000, (64, 4), generator=g, dtype=torch.int32)
    k = torch.full((64,), 4, dtype=torch.int32)
    out = wl.apply_boost(cfg, logits, drafts, k, wl.boost_probs(cfg), g)
    rows = torch.arange(64)[:, None]
    j = torch.arange(4)[None, :]
    changed = out[rows, j, drafts.long()] != logits[rows, j, drafts.long()]
    target = (logits[:, :4].float().amax(dim=-1) + 6.0).to(torch.bfloat16)
    assert torch.equal(out[rows, j, drafts.long()][changed], target[changed])
    assert 0.4 < changed.float().mean().item() < 0.6  # boost w.p. 0.5
    # nothing but the boosted entries moved
    diff = (out != logits).sum().item()
    assert diff == int(changed.sum().item())


def test_dense_drafts_follow_q():
    cfg = wl.get("c4", B=8, V=2000)
    g = wl._gen(4, "cpu")
    logits = wl.step_logits(cfg, g)
    q, d = wl.dense_draft(cfg, logits, g)
    assert q.shape == (8, 4, 2000) and q.dtype == torch.float32 and d.shape == (8, 4)
    assert torch.allclose(q.sum(-1), torch.ones(8, 4), atol=1e-5)
    assert (d >= 0).all() and (d < 2000).all()
    # the drafts are draws from q: their q values are large, far above uniform
    qd = q.gather(-1, d.long()[..., None])[..., 0]
    assert qd.mean().item() > 50.0 / 2000


def test_per_sequence_draft_caps_are_uniform():
    cfg = wl.get("c5", B=20000)
    k = wl.draft_limits(cfg, wl._gen(2, "cpu")).numpy()
    counts = np.bincount(k, minlength=5)
    assert k.min() == 0 and k.max() == 4
    assert np.abs(counts / k.size - 0.2).max() < 0.02
    assert (wl.draft_limits(wl.get("c3", B=10), wl._gen(2, "cpu")) == 4).all()


def test_generators_are_deterministic():
    cfg = wl.get("c5", B=3, V=4000, hist_len=(600, 600))
    a = wl.histories(cfg)
    b = wl.histories(cfg)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(wl.step_logits(cfg, wl._gen(1, "cpu")), wl.step_logits(cfg, wl._gen(1, "cpu")))
