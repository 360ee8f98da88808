"""GPU tests of the decode-step bookkeeping: the KV block pool against its
oracle, the device step counter, and a whole step captured in a CUDA graph
and replayed, against the same steps run eagerly."""
import numpy as np
import pytest
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from oracle import kv as okv

pytestmark = pytest.mark.gpu

KV_SHORT = 0x200


@pytest.fixture(autouse=True)
def _clean_status():
    sp.get_status(clear=True)
    yield


def _device_state(pool):
    top = int(pool.free_top.item())
    free = pool.free_stack[:top].cpu().tolist()
    nb = pool.nblocks.cpu().tolist()
    tab = pool.block_table.cpu().tolist()
    tables = [row[:n] for row, n in zip(tab, nb)]
    pads = [row[n:] for row, n in zip(tab, nb)]
    return free, tables, pads


def test_kv_pool_single_sequence_matches_oracle_exactly():
    # one sequence is served by one thread, so even the block ids are unique
    rng = np.random.default_rng(3)
    pool = sp.KvPool(num_blocks=40, B=1, max_blocks=16, block_size=4)
    ref = okv.KvPool(40, 1, 16, 4)
    kv = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvh = 0
    for it in range(60):
        op = rng.random()
        if op < 0.5:
            extra = int(rng.integers(0, 9))
            pool.reserve(kv, extra)
            ref.reserve([kvh], extra)
        elif op < 0.9:
            kvh = max(0, kvh + int(rng.integers(-6, 8)))
            kv.fill_(kvh)
            pool.trim(kv)
            ref.trim([kvh])
        else:
            pool.release(torch.ones(1, dtype=torch.int32, device="cuda"))
            ref.release([1])
        free, tables, pads = _device_state(pool)
        assert free == ref.free and tables == ref.tables, it
        assert all(x == -1 for row in pads for x in row)
        assert bool(sp.get_status() & KV_SHORT) == ref.short
        ref.short = False


@pytest.mark.parametrize("num_blocks", [2000, 150])
def test_kv_pool_many_sequences(num_blocks):
    # concurrent sequences: the counts are unique (the totals when the pool runs
    # short); every block is held by one sequence or free, exactly once
    rng = np.random.default_rng(num_blocks)
    B, mb, bs = 64, 24, 16
    pool = sp.KvPool(num_blocks=num_blocks, B=B, max_blocks=mb, block_size=bs)
    ref = okv.KvPool(num_blocks, B, mb, bs)
    kvh = rng.integers(0, 200, size=B)
    kv = torch.from_numpy(kvh.astype(np.int32)).cuda()
    for it in range(30):
        op = rng.random()
        if op < 0.5:
            pool.reserve(kv, 5)
            ref.reserve(kvh, 5)
        elif op < 0.85:
            kvh = np.maximum(0, kvh + rng.integers(-40, 30, size=B))
            kv.copy_(torch.from_numpy(kvh.astype(np.int32)))
            pool.trim(kv)
            ref.trim(kvh)
        else:
            done = (rng.random(B) < 0.2).astype(np.int32)
            pool.release(torch.from_numpy(done).cuda())
            ref.release(done)
        free, tables, pads = _device_state(pool)
        held = [x for t in tables for x in t]
        assert sorted(held + free) == list(range(num_blocks)), it
        assert all(x == -1 for row in pads for x in row)
        short = bool(sp.get_status() & KV_SHORT)
        assert short == ref.short, it
        if ref.short:
            assert sum(len(t) for t in tables) == sum(ref.counts()), it
            # re-synchronise the oracle with the device's choice of who got blocks
            ref.tables = [list(t) for t in tables]
            ref.free = list(free)
        else:
            assert [len(t) for t in tables] == ref.counts(), it
        ref.short = False


def test_pool_rejects_bad_sizes():
    with pytest.raises(sp.SpecngError):
        sp.KvPool(num_blocks=0, B=1, max_blocks=1, block_size=1)


def _small_path(seed=11, B=6, K=4, V=4096, cap=512):
    g = torch.Generator().manual_seed(seed)
    hist = torch.full((B, cap), -1, dtype=torch.int32)
    lens = torch.full((B,), 96, dtype=torch.int32)
    base = torch.randint(0, 4096, (B, 24), generator=g, dtype=torch.int32)
    for b in range(B):
        hist[b, :96] = base[b].repeat(4)  # a repeated span: the n-gram tables draft its continuation
    return hist, lens, base, g


def _copy_task_logits(base, lens, K1, V, g):
    """Target logits of one step that favour continuing each sequence's
    repeated span (so drafts are often accepted, and sometimes not)."""
    B, P = base.shape
    x = torch.randn((B, K1, V), generator=g) * 2
    for b in range(B):
        for j in range(K1):
            x[b, j, base[b, (int(lens[b]) + j) % P]] += 14.0
    return x


def _run(hist0, lens0, logits, use_graph, base=None, gen=None, steps=8, K=4, V=4096):
    B, cap = hist0.shape
    K1 = K + 1
    dev = "cuda"
    hist, lens = hist0.clone().to(dev), lens0.clone().to(dev)
    table = sp.NgramTable(B, V, B * cap)
    sp.ngram_update(table, hist, lens)
    drafts, k = sp.ngram_draft(table, hist, lens, K)
    kv = (lens + k + 1).to(torch.int32)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sp.spec_verify_workspace(B, K, V)
    pool = sp.KvPool(num_blocks=4096, B=B, max_blocks=64, block_size=16)
    pool.reserve(kv, 0)
    step_t = torch.zeros(1, dtype=torch.int64, device=dev)
    buf = torch.empty((B, K1, V), dtype=torch.float32, device=dev)
    params = sp.VerifyParams(temperature=1.0, rep_penalty=1.1, rep_window=16, gate_enabled=True, seed=5)

    def step(s):
        if use_graph:
            params.step_dev = step_t
        else:
            params.step = s
        sp.spec_verify(buf, drafts, None, k, hist, lens, params, kv, ema, out, acc, ws)
        sp.spec_commit(table, hist, lens, out, acc, K, out_drafts=drafts, out_k=k)
        pool.trim(kv)
        pool.reserve(kv, K + 1)
        if use_graph:
            sp.step_advance(step_t)

    rec = []
    if use_graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step(0)
    for s in range(steps):
        if len(logits) <= s:  # made from the current lengths (the eager run), then reused
            logits.append(_copy_task_logits(base, lens.cpu(), K1, V, gen))
        buf.copy_(logits[s])
        if use_graph:
            gr.replay()
        else:
            step(s)
        torch.cuda.synchronize()
        rec.append((out.cpu().clone(), acc.cpu().clone(), kv.cpu().clone(), ema.cpu().clone(),
                    drafts.cpu().clone(), k.cpu().clone(), lens.cpu().clone(), pool.nblocks.cpu().clone()))
    assert int(step_t.item()) == (steps if use_graph else 0)
    return rec, hist.cpu()


def test_step_replayed_from_cuda_graph_matches_eager():
    hist0, lens0, base, gen = _small_path()
    logits = []
    # the eager run first: it also takes the library's one-time setup before the capture
    eager, h_e = _run(hist0, lens0, logits, use_graph=False, base=base, gen=gen)
    graph, h_g = _run(hist0, lens0, logits, use_graph=True)
    assert sp.get_status() == 0
    for s, (a, b) in enumerate(zip(eager, graph)):
        for x, y in zip(a, b):
            assert torch.equal(x, y), s
    assert torch.equal(h_e, h_g)
    # the run exercised acceptances and rollbacks
    accs = torch.stack([r[1] for r in eager])
    assert int(accs.sum()) > 0 and int((accs == 0).sum()) > 0


def test_step_dev_equals_host_step():
    B, K, V = 5, 3, 3000
    g = torch.Generator().manual_seed(1)
    logits = torch.randn((B, K + 1, V), generator=g)
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32).cuda()
    k = torch.full((B,), K, dtype=torch.int32, device="cuda")
    outs = []
    for use_dev in (False, True):
        kv = torch.full((B,), 50, dtype=torch.int32, device="cuda")
        ema = torch.ones(B, device="cuda")
        out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        p = sp.VerifyParams(temperature=0.8, gate_enabled=False, seed=9, probe_interval=3)
        if use_dev:
            p.step_dev = torch.tensor([1234567], dtype=torch.int64, device="cuda")
        else:
            p.step = 1234567
        sp.spec_verify(logits.cuda(), drafts, None, k, None, None, p, kv, ema, out, acc,
                       sp.spec_verify_workspace(B, K, V))
        outs.append((out.cpu(), acc.cpu(), kv.cpu(), ema.cpu()))
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_step_dev_rejected_by_single_kernel_schedule():
    B, K, V = 2, 2, 1000
    p = sp.VerifyParams(temperature=1.0, schedule=1, step_dev=torch.zeros(1, dtype=torch.int64, device="cuda"))
    with pytest.raises(sp.SpecngError):
        sp.spec_verify(torch.randn(B, K + 1, V, device="cuda"), torch.zeros(B, K, dtype=torch.int32, device="cuda"),
                       None, torch.full((B,), K, dtype=torch.int32, device="cuda"), None, None, p,
                       torch.zeros(B, dtype=torch.int32, device="cuda"), torch.ones(B, device="cuda"),
                       torch.empty(B, K + 1, dtype=torch.int32, device="cuda"),
                       torch.empty(B, dtype=torch.int32, device="cuda"), sp.spec_verify_workspace(B, K, V))
