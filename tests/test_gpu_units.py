"""GPU unit tests: Philox bit-exactness, n-gram table against the oracle,
edge cases and device-detected faults (status bits; no GPU fault is made)."""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from oracle import ngram as on
from oracle import philox as op
from oracle import verify as ov

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    sp.get_status(clear=True)
    yield


def test_philox_bit_exact_on_1e6_counters():
    rng = np.random.default_rng(5)
    n = 1_000_000
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    for seed in (0, 0xDEADBEEFCAFEF00D):
        got = sp.philox4x32_10(torch.from_numpy(ctr.view(np.int32)).cuda(), seed).cpu().numpy().view(np.uint32)
        k0, k1 = op.seed_key(seed)
        ref = np.stack(op.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], k0, k1), axis=1)
        np.testing.assert_array_equal(got.astype(np.uint64), ref)


def _ngram_case(rng, B, V, L, cap):
    hist = np.full((B, cap), -1, dtype=np.int64)
    lens = rng.integers(0, L + 1, size=B)
    for b in range(B):
        hist[b, :lens[b]] = rng.integers(0, V, size=lens[b])
    return hist, lens


@pytest.mark.parametrize("seed", range(4))
def test_ngram_matches_oracle_incremental(seed):
    rng = np.random.default_rng(seed)
    B, V, cap = 37, 6, 400
    hist, lens = _ngram_case(rng, B, V, 120, cap)
    t = sp.NgramTable(B, V, B * cap)
    hg = torch.from_numpy(hist.astype(np.int32)).cuda()
    lg = torch.from_numpy(lens.astype(np.int32)).cuda()
    for rnd in range(6):
        sp.ngram_update(t, hg, lg)
        for max_k in (0, 1, 4, 9):
            lim = torch.from_numpy(rng.integers(0, 10, size=B).astype(np.int32)).cuda()
            for k_limit in (None, lim):
                d, k = sp.ngram_draft(t, hg, lg, max_k, k_limit=k_limit)
                kl = None if k_limit is None else k_limit.cpu().numpy()
                d_o, k_o = on.draft_batch(hist, lens, max_k, k_limit=kl)
                np.testing.assert_array_equal(k.cpu().numpy(), k_o)
                np.testing.assert_array_equal(d.cpu().numpy(), d_o)
        grow = rng.integers(0, 30, size=B)
        for b in range(B):
            n = min(grow[b], cap - lens[b])
            hist[b, lens[b]:lens[b] + n] = rng.integers(0, V, size=n)
            lens[b] += n
        hg.copy_(torch.from_numpy(hist.astype(np.int32)))
        lg.copy_(torch.from_numpy(lens.astype(np.int32)))
    assert sp.get_status() == 0
    # a table rebuilt in one update drafts the same as the incremental one
    t2 = sp.NgramTable(B, V, B * cap)
    sp.ngram_update(t, hg, lg)
    sp.ngram_update(t2, hg, lg)
    a = sp.ngram_draft(t, hg, lg, 8)
    b_ = sp.ngram_draft(t2, hg, lg, 8)
    assert torch.equal(a[0], b_[0]) and torch.equal(a[1], b_[1])
    t.reset()
    sp.ngram_update(t, hg, lg)
    c = sp.ngram_draft(t, hg, lg, 8)
    assert torch.equal(a[0], c[0])


def test_ngram_fallback_pads_to_the_cap():
    rng = np.random.default_rng(4)
    B, V, cap = 40, 7, 200
    hist, lens = _ngram_case(rng, B, V, 60, cap)
    t = sp.NgramTable(B, V, B * cap)
    hg = torch.from_numpy(hist.astype(np.int32)).cuda()
    lg = torch.from_numpy(lens.astype(np.int32)).cuda()
    sp.ngram_update(t, hg, lg)
    fb = rng.integers(0, V, size=(B, 5))
    lim = rng.integers(0, 6, size=B)
    d, k = sp.ngram_draft(t, hg, lg, 5, k_limit=torch.from_numpy(lim.astype(np.int32)).cuda(),
                          fallback=torch.from_numpy(fb.astype(np.int32)).cuda())
    d_o, k_o = on.draft_batch(hist, lens, 5, k_limit=lim, fallback=fb)
    np.testing.assert_array_equal(k.cpu().numpy(), lim)
    np.testing.assert_array_equal(k.cpu().numpy(), k_o)
    np.testing.assert_array_equal(d.cpu().numpy(), d_o)


def test_ngram_fallback_after_a_miss_part_way():
    # the table indexes the prefix [1, 2, 3] while the history has grown to
    # [1, 2, 3, 9, 1] (no update since): the chain drafts 2, 3 and then misses,
    # so positions 2.. of the cap take fallback[b, 2:k_b] (worked by hand in
    # tests/test_oracle_ngram.py)
    B, V = 5, 64
    hist = torch.full((B, 8), -1, dtype=torch.int32)
    hist[:, :5] = torch.tensor([1, 2, 3, 9, 1], dtype=torch.int32)
    t = sp.NgramTable(B, V, B * 8)
    hg = hist.cuda()
    sp.ngram_update(t, hg, torch.full((B,), 3, dtype=torch.int32, device="cuda"))
    lens = torch.full((B,), 5, dtype=torch.int32, device="cuda")
    fb = torch.tensor([[40, 41, 42, 43]] * B, dtype=torch.int32, device="cuda")
    lim = torch.tensor([4, 3, 2, 1, 0], dtype=torch.int32, device="cuda")
    d, k = sp.ngram_draft(t, hg, lens, 4, k_limit=lim, fallback=fb)
    want = [[2, 3, 42, 43], [2, 3, 42, -1], [2, 3, -1, -1], [2, -1, -1, -1], [-1, -1, -1, -1]]
    assert d.cpu().tolist() == want
    assert k.cpu().tolist() == [4, 3, 2, 1, 0]
    assert sp.get_status() == 0


def test_ngram_large_vocab_keys():
    # ids near 2^18 exercise every key field
    rng = np.random.default_rng(9)
    B, V, cap = 512, 262144, 64
    hist = np.full((B, cap), -1, dtype=np.int64)
    lens = np.full(B, cap)
    base = rng.integers(V - 8, V, size=(B, cap))
    hist[:, :] = base
    t = sp.NgramTable(B, V, B * cap)
    hg = torch.from_numpy(hist.astype(np.int32)).cuda()
    lg = torch.from_numpy(lens.astype(np.int32)).cuda()
    sp.ngram_update(t, hg, lg)
    d, k = sp.ngram_draft(t, hg, lg, 4)
    d_o, k_o = on.draft_batch(hist, lens, 4)
    np.testing.assert_array_equal(d.cpu().numpy(), d_o)
    np.testing.assert_array_equal(k.cpu().numpy(), k_o)
    assert sp.get_status() == 0


def test_table_full_sets_status_and_returns():
    B, V, cap = 4, 50000, 2000
    rng = np.random.default_rng(1)
    hist = torch.from_numpy(rng.integers(0, V, size=(B, cap)).astype(np.int32)).cuda()
    lens = torch.full((B,), cap, dtype=torch.int32, device="cuda")
    t = sp.NgramTable(B, V, 64)   # 1024 slots for 8000 distinct pairs
    assert t.capacity == 1024
    sp.ngram_update(t, hist, lens)
    sp.ngram_draft(t, hist, lens, 4)
    bits = sp.get_status()
    assert bits & 0x01


def test_out_of_range_tokens_set_status():
    B, V = 2, 100
    hist = torch.tensor([[1, 2, 3, 500, 4, 5, 6, 7], [1, -3, 2, 2, 2, 2, 2, 2]], dtype=torch.int32, device="cuda")
    lens = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    t = sp.NgramTable(B, V, 64)
    sp.ngram_update(t, hist, lens)
    assert sp.get_status() & 0x02


def test_append_overflow_and_bad_accept():
    hist = torch.zeros((2, 10), dtype=torch.int32, device="cuda")
    lens = torch.tensor([8, 2], dtype=torch.int32, device="cuda")
    out = torch.tensor([[1, 2, 3], [4, 5, 6]], dtype=torch.int32, device="cuda")
    acc = torch.tensor([2, 1], dtype=torch.int32, device="cuda")
    sp.spec_append(hist, lens, out, acc)
    assert sp.get_status() & 0x08
    assert lens.tolist() == [8, 4] and hist[1, 2:4].tolist() == [4, 5]
    acc = torch.tensor([5, 0], dtype=torch.int32, device="cuda")
    sp.spec_append(hist, lens, out, acc)
    assert sp.get_status() & 0x10
    assert lens.tolist() == [8, 5]


def _verify(logits, drafts, k, params, q=None, hist=None, lens=None):
    B, K1, V = logits.shape
    dev = "cuda"
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K1 - 1, V)
    sp.spec_verify(logits.cuda(), drafts.cuda(), None if q is None else q.cuda(), k.cuda(),
                   None if hist is None else hist.cuda(), None if lens is None else lens.cuda(),
                   params, kv, ema, out, acc, ws)
    return out.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy(), ema.cpu().numpy()


def test_nonfinite_logits_set_status():
    logits = torch.randn(2, 3, 1000)
    logits[1, 0, 17] = float("nan")
    logits[0, 0, 3] = float("inf")
    _verify(logits, torch.zeros(2, 2, dtype=torch.int32), torch.tensor([2, 2], dtype=torch.int32),
            sp.VerifyParams(temperature=1.0, gate_enabled=False))
    assert sp.get_status() & 0x04


def test_bad_k_and_bad_draft_set_status():
    logits = torch.randn(2, 3, 1000)
    _verify(logits, torch.tensor([[1, 2], [5000, 1]], dtype=torch.int32), torch.tensor([7, 2], dtype=torch.int32),
            sp.VerifyParams(temperature=1.0, gate_enabled=False))
    bits = sp.get_status()
    assert bits & 0x10 and bits & 0x02


def test_misaligned_logits_pointer_uses_scalar_path():
    # a view starting 2 bytes into the buffer cannot take 16-byte loads
    B, K, V = 3, 2, 20000
    g = torch.Generator().manual_seed(3)
    base = (torch.randn(B * (K + 1) * V + 1, generator=g) * 4).to(torch.bfloat16)
    logits = base[1:].view(B, K + 1, V)
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    k = torch.tensor([2, 1, 0], dtype=torch.int32)
    p = sp.VerifyParams(temperature=0.7, gate_enabled=False, seed=5, step=2)
    gpu = torch.empty(B * (K + 1) * V + 1, dtype=torch.bfloat16, device="cuda")
    gpu.copy_(base)
    lg = gpu[1:].view(B, K + 1, V)
    assert lg.data_ptr() % 16 != 0
    kv = torch.full((B,), 100, dtype=torch.int32, device="cuda")
    ema = torch.ones(B, dtype=torch.float32, device="cuda")
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    acc = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = sp.spec_verify_workspace(B, K, V)
    sp.spec_verify(lg, drafts.cuda(), None, k.cuda(), None, None, p, kv, ema, out, acc, ws)
    res = ov.spec_verify(logits.float().numpy(), drafts.numpy(), None, k.numpy(), np.zeros((B, 1), int),
                         np.zeros(B, int), ov.VerifyParams(temperature=0.7, gate_enabled=False, seed=5, step=2),
                         np.full(B, 100), np.ones(B))
    np.testing.assert_array_equal(out.cpu().numpy(), res["out_tokens"])
    np.testing.assert_array_equal(acc.cpu().numpy(), res["accept_len"])


def test_workspace_is_reusable_across_shapes_and_calls():
    # tickets reset themselves: many calls on one workspace, different B/K/V within its size
    ws = sp.spec_verify_workspace(8, 4, 50000)
    g = torch.Generator().manual_seed(0)
    for it, (B, K, V) in enumerate([(8, 4, 50000), (3, 2, 777), (8, 4, 50000), (1, 0, 10), (5, 4, 33333)]):
        logits = torch.randn(B, K + 1, V, generator=g) * 3
        drafts = torch.randint(0, V, (B, max(K, 1)), generator=g, dtype=torch.int32)[:, :K].contiguous()
        k = torch.full((B,), K, dtype=torch.int32)
        p = sp.VerifyParams(temperature=1.0, gate_enabled=False, seed=it, step=it)
        kv = torch.full((B,), 50, dtype=torch.int32, device="cuda")
        ema = torch.ones(B, dtype=torch.float32, device="cuda")
        out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        acc = torch.empty((B,), dtype=torch.int32, device="cuda")
        sp.spec_verify(logits.cuda(), drafts.cuda(), None, k.cuda(), None, None, p, kv, ema, out, acc, ws)
        res = ov.spec_verify(logits.numpy(), drafts.numpy().reshape(B, K), None, k.numpy(),
                             np.zeros((B, 1), int), np.zeros(B, int),
                             ov.VerifyParams(temperature=1.0, gate_enabled=False, seed=it, step=it),
                             np.full(B, 50), np.ones(B))
        np.testing.assert_array_equal(out.cpu().numpy(), res["out_tokens"])
    assert sp.get_status() == 0


def test_all_gated_reads_only_row_zero():
    # with every sequence gated off, rows >= 1 are never read: poison them
    B, K, V = 4, 4, 5000
    logits = torch.randn(B, K + 1, V) * 2
    logits[:, 1:] = float("nan")
    drafts = torch.randint(0, V, (B, K), dtype=torch.int32)
    k = torch.full((B,), K, dtype=torch.int32)
    dev = "cuda"
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.full((B,), 0.3, dtype=torch.float32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K, V)
    p = sp.VerifyParams(temperature=1.0, gate_enabled=True, seed=1)
    sp.spec_verify(logits.cuda(), drafts.cuda(), None, k.cuda(), None, None, p, kv, ema, out, acc, ws)
    assert sp.get_status() == 0
    assert (acc.cpu() == 0).all() and (kv.cpu() == 100 - K).all()
    assert torch.allclose(ema.cpu(), torch.full((B,), 0.3))
    res = ov.spec_verify(logits[:, :1].numpy(), np.zeros((B, 0), int), None, np.zeros(B, int),
                         np.zeros((B, 1), int), np.zeros(B, int),
                         ov.VerifyParams(temperature=1.0, gate_enabled=False, seed=1), np.zeros(B), np.ones(B))
    np.testing.assert_array_equal(out.cpu().numpy()[:, 0], res["out_tokens"][:, 0])


@pytest.mark.parametrize("seed", range(3))
def test_commit_equals_append_update_draft(seed):
    # spec_commit against the three calls it fuses, over several steps, and the
    # drafts against the oracle on the resulting histories
    rng = np.random.default_rng(100 + seed)
    B, V, K, cap = 29, 9, 4, 300
    hist, lens = _ngram_case(rng, B, V, 80, cap)
    t1, t2 = sp.NgramTable(B, V, B * cap), sp.NgramTable(B, V, B * cap)
    h1 = torch.from_numpy(hist.astype(np.int32)).cuda()
    l1 = torch.from_numpy(lens.astype(np.int32)).cuda()
    h2, l2 = h1.clone(), l1.clone()
    sp.ngram_update(t1, h1, l1)
    sp.ngram_update(t2, h2, l2)
    for step in range(8):
        a = torch.from_numpy(rng.integers(0, K + 1, size=B).astype(np.int32)).cuda()
        if step == 5:
            a.fill_(K)  # the longest history cannot take K + 1 more tokens below this step's cap
        tok = torch.from_numpy(rng.integers(0, V, size=(B, K + 1)).astype(np.int32)).cuda()
        lim = torch.from_numpy(rng.integers(0, K + 1, size=B).astype(np.int32)).cuda() if step % 2 else None
        fb = torch.from_numpy(rng.integers(0, V, size=(B, K)).astype(np.int32)).cuda() if step % 3 == 0 else None
        cap_now = cap if step != 5 else int(l1.max().item()) + 2   # some sequences overflow at step 5
        sp.spec_append(h1, l1, tok, a, hist_cap=cap_now)
        sp.ngram_update(t1, h1, l1)
        d1, k1 = sp.ngram_draft(t1, h1, l1, K, k_limit=lim, fallback=fb)
        d2, k2 = sp.spec_commit(t2, h2, l2, tok, a, K, k_limit=lim, fallback=fb, hist_cap=cap_now)
        assert torch.equal(h1, h2) and torch.equal(l1, l2)
        assert torch.equal(d1, d2) and torch.equal(k1, k2)
        d_o, k_o = on.draft_batch(h2.cpu().numpy().astype(np.int64), l2.cpu().numpy().astype(np.int64), K,
                                  k_limit=None if lim is None else lim.cpu().numpy(),
                                  fallback=None if fb is None else fb.cpu().numpy())
        np.testing.assert_array_equal(d2.cpu().numpy(), d_o)
        np.testing.assert_array_equal(k2.cpu().numpy(), k_o)
    assert sp.status_names(sp.get_status()) == ["HIST_OVERFLOW"]


@pytest.mark.parametrize("rep", [1.0, 1.3])
def test_all_zero_residual_falls_back_to_p(rep):
    # q >= p everywhere (p rounded up to fp32) and q(d) = 1 at a draft of tiny p: the
    # draft is rejected and the residual max(0, p - q) is zero everywhere, so the
    # token is the Gumbel-max sample of p at that row (the oracle's fallback rule)
    B, K, V, T = 4, 2, 5000, 0.7
    g = torch.Generator().manual_seed(11)
    logits = torch.randn(B, K + 1, V, generator=g) * 3
    hist = torch.randint(0, V, (B, 40), generator=g, dtype=torch.int32)
    lens = torch.full((B,), 40, dtype=torch.int32)
    kw = dict(temperature=T, rep_penalty=rep, rep_window=16 if rep != 1.0 else 0, gate_enabled=False, seed=9, step=4)
    op_ = ov.VerifyParams(**kw)
    drafts = torch.zeros((B, K), dtype=torch.int32)
    # drafts of tiny p, chosen row by row (the penalty window of row j covers the drafts before it)
    for j in range(K):
        zj = ov.transform_rows(logits.numpy().astype(np.float64), op_, hist.numpy(), lens.numpy(), drafts.numpy())
        drafts[:, j] = torch.from_numpy(np.argmin(zj[:, j], axis=-1).astype(np.int32))
    z = ov.transform_rows(logits.numpy().astype(np.float64), op_, hist.numpy(), lens.numpy(), drafts.numpy())
    p = np.exp(ov.log_softmax(z[:, :K] / op_.f64("temperature")))
    q = p.astype(np.float32)
    q = np.where(q.astype(np.float64) < p, np.nextafter(q, np.float32(np.inf)), q).astype(np.float32)
    q[np.arange(B)[:, None], np.arange(K)[None, :], drafts.numpy()] = 1.0
    assert (q.astype(np.float64) >= p).all()
    k = torch.full((B,), K, dtype=torch.int32)
    dev = "cuda"
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K, V)
    sp.spec_verify(logits.cuda(), drafts.cuda(), torch.from_numpy(q).cuda(), k.cuda(), hist.cuda(), lens.cuda(),
                   sp.VerifyParams(**kw), kv, ema, out, acc, ws)
    res = ov.spec_verify(logits.numpy(), drafts.numpy(), q, k.numpy(), hist.numpy(), lens.numpy(), op_,
                         np.full(B, 100), np.ones(B))
    assert (res["accept_len"] == 0).all()
    np.testing.assert_array_equal(acc.cpu().numpy(), res["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), res["out_tokens"])
    assert sp.get_status() == 0


def test_sixteen_drafts_every_warp_testing():
    # K = 16: every warp of the decision kernel takes an accept test, none is free
    # to prepare row 0 early; the row must then be prepared after the tests
    B, K, V = 3, 16, 5000
    g = torch.Generator().manual_seed(21)
    logits = torch.randn(B, K + 1, V, generator=g) * 3
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    k = torch.full((B,), K, dtype=torch.int32)
    kw = dict(temperature=0.8, gate_enabled=False, seed=4, step=9)
    dev = "cuda"
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K, V)
    sp.spec_verify(logits.cuda(), drafts.cuda(), None, k.cuda(), None, None, sp.VerifyParams(**kw), kv, ema, out,
                   acc, ws)
    res = ov.spec_verify(logits.numpy(), drafts.numpy(), None, k.numpy(), np.zeros((B, 1), int), np.zeros(B, int),
                         ov.VerifyParams(**kw), np.full(B, 100), np.ones(B))
    np.testing.assert_array_equal(acc.cpu().numpy(), res["accept_len"])
    np.testing.assert_array_equal(out.cpu().numpy(), res["out_tokens"])
    assert sp.get_status() == 0
