"""Fused LM head + verify (spec_verify_lmhead) against the oracle.

The parity cases draw the hidden states and the head's weight from a grid
(integers in [-2, 2] / 16, exact in bf16): every dot product and every fp32
partial sum of it is then exact, whatever the order of the tensor cores'
accumulation, so the logits (each rounded once to bf16) and every decision
taken on them are compared bit for bit with the oracle.  A case with
Gaussian inputs checks the GEMM alone within its rounding bound.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from oracle import lmhead as ol
from oracle import verify as ov


@pytest.fixture(autouse=True)
def _clean_status(request):
    if request.node.get_closest_marker("gpu") is not None:
        sp.get_status(clear=True)
    yield


def _grid(g, shape):
    return (torch.randint(-2, 3, shape, generator=g).float() / 16).to(torch.bfloat16)


def _case(B, K, V, d, seed, argmax_drafts=0.5):
    """hidden, weight (bf16, CPU), the oracle's logits (fp64) and drafts: each
    d_{j+1} the argmax of row j w.p. argmax_drafts (so some drafts are accepted)."""
    g = torch.Generator().manual_seed(seed)
    hidden = _grid(g, (B, K + 1, d))
    weight = _grid(g, (V, d))
    ref = ol.lm_head_logits(hidden.float().numpy(), weight.float().numpy())
    rnd = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32).numpy()
    coin = torch.rand((B, K), generator=g).numpy() < argmax_drafts
    am = ref[:, :K].argmax(-1)
    drafts = np.where(coin, am, rnd).astype(np.int32)
    k = torch.randint(0, K + 1, (B,), generator=g, dtype=torch.int32).numpy()
    return hidden, weight, ref, drafts, k


def _run_gpu(hidden, weight, drafts, k, kw, q=None, ema0=1.0):
    B, K1, d = hidden.shape
    V = weight.shape[0]
    dev = "cuda"
    logits = torch.empty((B, K1, V), dtype=torch.bfloat16, device=dev)
    kv = torch.full((B,), 100, dtype=torch.int32, device=dev)
    ema = torch.full((B,), ema0, dtype=torch.float32, device=dev)
    out = torch.empty((B, K1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_lmhead_workspace(B, K1 - 1, V)
    sp.spec_verify_lmhead(hidden.cuda(), weight.cuda(), logits, torch.from_numpy(drafts).cuda(),
                          None if q is None else torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(),
                          None, None, sp.VerifyParams(**kw), kv, ema, out, acc, ws)
    torch.cuda.synchronize()
    return logits, out.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy(), ema.cpu().numpy()


def _check(ref, drafts, k, kw, got, q=None, ema0=1.0, rows=None):
    logits, out, acc, kv, ema = got
    B = ref.shape[0]
    res = ov.spec_verify(ref, drafts, q, k, np.zeros((B, 1), int), np.zeros(B, int), ov.VerifyParams(**kw),
                         np.full(B, 100), np.full(B, ema0))
    np.testing.assert_array_equal(logits.float().cpu().numpy(), ref)
    np.testing.assert_array_equal(acc, res["accept_len"])
    np.testing.assert_array_equal(out, res["out_tokens"])
    np.testing.assert_array_equal(kv, res["kv_len"])
    np.testing.assert_allclose(ema, res["ema"], atol=1e-6)
    assert sp.get_status() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("kw", [
    dict(temperature=0.7, gate_enabled=False, seed=3, step=1),
    dict(temperature=0.0, gate_enabled=False, seed=3, step=1),
    dict(temperature=1.0, softcap=30.0, gate_enabled=True, seed=9, step=4),
])
def test_small_ragged_shapes(kw):
    # 15 rows (one partial row tile), V = 1032 (four whole vocab tiles and one of 8 ids), d = 128
    hidden, weight, ref, drafts, k = _case(3, 4, 1032, 128, seed=1)
    _check(ref, drafts, k, kw, _run_gpu(hidden, weight, drafts, k, kw))


@pytest.mark.gpu
@pytest.mark.parametrize("kw", [
    dict(temperature=0.6, gate_enabled=False, seed=5, step=2),
    dict(temperature=0.0, gate_enabled=False, seed=5, step=2),
])
def test_several_tiles(kw):
    # 200 rows (two row tiles), 17 vocab tiles, d = 256 (four stages of the ring)
    hidden, weight, ref, drafts, k = _case(40, 4, 4104, 256, seed=2)
    _check(ref, drafts, k, kw, _run_gpu(hidden, weight, drafts, k, kw))


@pytest.mark.gpu
def test_dense_draft_distributions():
    B, K, V, d = 8, 4, 2056, 192
    hidden, weight, ref, drafts, k = _case(B, K, V, d, seed=4)
    rng = np.random.default_rng(4)
    q = rng.random((B, K, V)).astype(np.float32) ** 8
    q /= q.sum(-1, keepdims=True)
    kw = dict(temperature=0.6, gate_enabled=False, seed=7, step=3)
    _check(ref, drafts, k, kw, _run_gpu(hidden, weight, drafts, k, kw, q=q), q=q)


@pytest.mark.gpu
def test_full_vocab_and_batch_sampled_sequences():
    # the c5 shape (B = 256, K = 4, V = 151936) with d = 512: the whole tile grid
    # (10 row tiles x 594 vocab tiles); the oracle checks four sequences
    B, K, V, d = 256, 4, 151936, 512
    g = torch.Generator().manual_seed(11)
    hidden = _grid(g, (B, K + 1, d))
    weight = _grid(g, (V, d))
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32).numpy()
    k = torch.randint(0, K + 1, (B,), generator=g, dtype=torch.int32).numpy()
    kw = dict(temperature=0.6, gate_enabled=False, seed=1, step=6)
    logits, out, acc, kv, ema = _run_gpu(hidden, weight, drafts, k, kw)
    wf = weight.float().numpy()
    for b in (0, 97, 128, 255):
        ref = ol.lm_head_logits(hidden[b:b + 1].float().numpy(), wf)
        np.testing.assert_array_equal(logits[b:b + 1].float().cpu().numpy(), ref)
        res = ov.spec_verify(ref, drafts[b:b + 1], None, k[b:b + 1], np.zeros((1, 1), int), np.zeros(1, int),
                             ov.VerifyParams(**kw), np.full(1, 100), np.ones(1), seq_ids=np.array([b]))
        assert acc[b] == res["accept_len"][0]
        np.testing.assert_array_equal(out[b], res["out_tokens"][0])
        assert kv[b] == res["kv_len"][0]
    assert sp.get_status() == 0


@pytest.mark.gpu
def test_many_row_tiles_and_a_partial_last_vocab_tile():
    # 153 row tiles (odd: single CTAs) on 152 SMs and V = 264 (a second vocab tile of 8 ids):
    # some CTAs run two tiles of the last vocab column one after the other, whose trailing
    # boxes lie past V; every logit and a sample of sequences' tokens against the oracle
    B, K, V, d = 19584, 0, 264, 64
    g = torch.Generator().manual_seed(13)
    hidden = _grid(g, (B, K + 1, d))
    weight = _grid(g, (V, d))
    drafts = np.zeros((B, 1), dtype=np.int32)
    k = np.zeros(B, dtype=np.int32)
    kw = dict(temperature=0.7, gate_enabled=False, seed=2, step=5)
    logits, out, acc, kv, ema = _run_gpu(hidden, weight, drafts[:, :0], k, kw)
    ref = ol.lm_head_logits(hidden.float().numpy(), weight.float().numpy())
    np.testing.assert_array_equal(logits.float().cpu().numpy(), ref)
    for b in (0, 1, 153, 19583):
        res = ov.spec_verify(ref[b:b + 1], drafts[b:b + 1, :0], None, k[b:b + 1], np.zeros((1, 1), int),
                             np.zeros(1, int), ov.VerifyParams(**kw), np.full(1, 100), np.ones(1), seq_ids=np.array([b]))
        np.testing.assert_array_equal(out[b], res["out_tokens"][0])
    assert sp.get_status() == 0


@pytest.mark.gpu
def test_gaussian_inputs_within_rounding():
    # the GEMM alone: fp32 accumulation, then one rounding to bf16.  Against the
    # fp64 product rounded once: one bf16 ulp (the fp32 error can move a value
    # across a rounding boundary) plus the summation bound d 2^-24 sum |h_i w_i|
    # (it dominates where the terms cancel and the result is small)
    B, K, V, d = 4, 4, 8192, 2560
    g = torch.Generator().manual_seed(12)
    hidden = (torch.randn(B, K + 1, d, generator=g)).to(torch.bfloat16)
    weight = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16)
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32).numpy()
    k = np.full(B, K, dtype=np.int32)
    logits, *_ = _run_gpu(hidden, weight, drafts, k, dict(temperature=1.0, gate_enabled=False))
    ref = ol.lm_head_logits(hidden.float().numpy(), weight.float().numpy())
    got = logits.float().cpu().numpy()
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    acc = d * 2.0 ** -24 * (np.abs(hidden.float().numpy()) @ np.abs(weight.float().numpy()).T)
    assert np.all(np.abs(got - ref) <= ulp + acc)
    assert np.mean(got == ref) > 0.99


def test_lmhead_rejects_what_it_does_not_support():
    # host-side checks, before any CUDA call: run without a GPU
    import ctypes
    from speculative_decoding_draft_ngram_gb300 import capi
    L = capi.load()
    p = sp.VerifyParams(temperature=1.0, rep_penalty=1.1, rep_window=8).to_c()
    buf = ctypes.c_void_p(256)  # never dereferenced: the checks fail first
    rc = L.spec_verify_lmhead(buf, buf, 64, buf, 1, 1, 64, buf, None, buf, buf, 8, buf, ctypes.byref(p),
                              buf, buf, buf, buf, buf, 1 << 20, None)
    assert rc == -1  # SPECNG_EINVAL: the repetition penalty
    p = sp.VerifyParams(temperature=1.0).to_c()
    rc = L.spec_verify_lmhead(buf, buf, 100, buf, 1, 1, 64, buf, None, buf, None, 0, None, ctypes.byref(p),
                              buf, buf, buf, buf, buf, 1 << 20, None)
    assert rc == -1  # d not a multiple of 64
    rc = L.spec_verify_lmhead(buf, buf, 64, buf, 1, 1, 60, buf, None, buf, None, 0, None, ctypes.byref(p),
                              buf, buf, buf, buf, buf, 1 << 20, None)
    assert rc == -1  # V not a multiple of 8


def test_lmhead_host_checks_null_alignment_schedule_and_workspace_size():
    # host-side checks that run before any CUDA call (no GPU needed)
    import ctypes
    from speculative_decoding_draft_ngram_gb300 import capi
    L = capi.load()
    p = sp.VerifyParams(temperature=1.0).to_c()
    ok = ctypes.c_void_p(4096)
    bad = ctypes.c_void_p(4096 + 8)   # 8-byte aligned only
    args = lambda h, w, d, lg: (h, w, d, lg, 1, 1, 64, ok, None, ok, None, 0, None, ctypes.byref(p),
                                ok, ok, ok, ok, ok, 1 << 20, None)
    assert L.spec_verify_lmhead(*args(None, ok, 64, ok)) == -1          # NULL hidden
    assert L.spec_verify_lmhead(*args(bad, ok, 64, ok)) == -2           # SPECNG_EALIGN
    assert L.spec_verify_lmhead(*args(ok, ok, 64, bad)) == -2
    assert L.spec_verify_lmhead(*args(ok, ok, (1 << 20) + 64, ok)) == -1  # d out of range
    pf = sp.VerifyParams(temperature=1.0, schedule=1).to_c()
    a = list(args(ok, ok, 64, ok))
    a[13] = ctypes.byref(pf)
    assert L.spec_verify_lmhead(*a) == -1                                # single-kernel schedule
    # the workspace: one 8-byte record per row and noise block beyond spec_verify's per-segment records
    B, K, V = 8, 4, 151936
    assert sp.spec_verify_lmhead_workspace_bytes(B, K, V) > sp.spec_verify_workspace_bytes(B, K, V)
    assert sp.spec_verify_lmhead_workspace_bytes(B, K, V) % 256 == 0
    assert sp.spec_verify_lmhead_workspace_bytes(0, K, V) == 0
