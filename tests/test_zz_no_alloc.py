"""spec_verify_noalloc (the library's static scratch instead of a caller
workspace) against spec_verify with a workspace: two calls in a row, the
second fed by the first's kv_len / ema, on point-mass, dense-q and greedy
inputs.  Both entry points run the same kernels, so every output must be
identical.  The file is named to be collected last, and each test sets up
its own state, so it passes alone and after the rest of the suite."""
import ctypes

import pytest
import torch

import speculative_decoding_draft_ngram_gb300 as sp
from speculative_decoding_draft_ngram_gb300 import capi


def _inputs(B, K, V, dense, seed):
    g = torch.Generator().manual_seed(seed)
    logits = [(torch.randn(B, K + 1, V, generator=g) * 4).to(torch.bfloat16) for _ in range(2)]
    drafts = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    k = torch.randint(0, K + 1, (B,), generator=g, dtype=torch.int32)
    q = None
    if dense:
        q = [torch.softmax(x[:, :K].float() / 0.6 + torch.randn(B, K, V, generator=g) * 0.5, dim=-1)
             for x in logits]
        k = torch.full((B,), K, dtype=torch.int32)
    hist = torch.randint(0, V, (B, 300), generator=g, dtype=torch.int32)
    lens = torch.full((B,), 290, dtype=torch.int32)
    return logits, drafts, k, q, hist, lens


def _two_calls(fn, B, K, V, dense, T, seed, with_ws):
    logits, drafts, k, q, hist, lens = _inputs(B, K, V, dense, seed)
    dev = "cuda"
    kv = torch.full((B,), 500, dtype=torch.int32, device=dev)
    ema = torch.full((B,), 0.55, dtype=torch.float32, device=dev)
    ws = sp.spec_verify_workspace(B, K, V) if with_ws else None
    outs = []
    for step in (1, 2):
        p = sp.VerifyParams(temperature=T, rep_penalty=1.1, rep_window=64, gate_enabled=True, seed=seed, step=step)
        out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        acc = torch.empty((B,), dtype=torch.int32, device=dev)
        args = (logits[step - 1].to(dev), drafts.to(dev), None if q is None else q[step - 1].to(dev), k.to(dev),
                hist.to(dev), lens.to(dev), p, kv, ema, out, acc)
        if with_ws:
            fn(*args, ws)
        else:
            fn(*args)
        outs.append((out.cpu(), acc.cpu(), kv.cpu(), ema.cpu()))
    return outs


CASES = {
    "point_mass_t06": (7, 4, 40000, False, 0.6),
    "dense_q_t06": (5, 4, 40001, True, 0.6),
    "greedy": (6, 3, 30000, False, 0.0),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point(name):
    B, K, V, dense, T = CASES[name]
    ref = _two_calls(sp.spec_verify, B, K, V, dense, T, 11, True)
    got = _two_calls(sp.spec_verify_noalloc, B, K, V, dense, T, 11, False)
    for (o1, a1, k1, e1), (o2, a2, k2, e2) in zip(ref, got):
        assert torch.equal(o1, o2)
        assert torch.equal(a1, a2)
        assert torch.equal(k1, k2)
        assert torch.equal(e1, e2)
    assert sp.get_status() == 0


@pytest.mark.gpu
def test_noalloc_leaves_free_device_memory_unchanged():
    B, K, V = 4, 4, 20000
    _two_calls(sp.spec_verify_noalloc, B, K, V, False, 0.6, 3, False)  # set-up: address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    logits, drafts, k, q, hist, lens = _inputs(B, K, V, False, 5)
    dev = "cuda"
    args = [x.to(dev) for x in (logits[0], drafts, k, hist, lens)]
    kv = torch.full((B,), 500, dtype=torch.int32, device=dev)
    ema = torch.ones(B, dtype=torch.float32, device=dev)
    out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    for step in range(5):
        p = sp.VerifyParams(temperature=0.6, gate_enabled=False, seed=1, step=step)
        sp.spec_verify_noalloc(args[0], args[1], None, args[2], args[3], args[4], p, kv, ema, out, acc)
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert free2 == free1, (free0, free1, free2)


@pytest.mark.gpu
def test_noalloc_near_the_scratch_limit():
    # B=740, K=4, V=262144 needs over 15.5 MiB of the 16 MiB scratch; the inputs
    # are made on the device (1.9 GB of bf16 logits), two calls in a row as above
    B, K, V = 740, 4, 262144
    need = sp.spec_verify_workspace_bytes(B, K, V)
    assert 15.5 * 2**20 < need <= 16 << 20
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(7)
    logits = (torch.randn((B, K + 1, V), generator=g, device=dev) * 8).to(torch.bfloat16)
    drafts = torch.randint(0, V, (B, K), generator=g, device=dev, dtype=torch.int32)
    k = torch.randint(0, K + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    results = []
    for fn, ws in ((sp.spec_verify, sp.spec_verify_workspace(B, K, V)), (sp.spec_verify_noalloc, None)):
        kv = torch.full((B,), 900, dtype=torch.int32, device=dev)
        ema = torch.full((B,), 0.6, dtype=torch.float32, device=dev)
        outs = []
        for step in (1, 2):
            p = sp.VerifyParams(temperature=1.0, softcap=30.0, gate_enabled=True, seed=3, step=step)
            out = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
            acc = torch.empty((B,), dtype=torch.int32, device=dev)
            args = (logits, drafts, None, k, None, None, p, kv, ema, out, acc)
            fn(*args, ws) if ws is not None else fn(*args)
            outs.append((out.cpu(), acc.cpu(), kv.cpu(), ema.cpu()))
        results.append(outs)
    for a, b in zip(*results):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    assert sp.get_status() == 0


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # host-side check, before any CUDA call: runs without a GPU
    from speculative_decoding_draft_ngram_gb300 import build as b
    b.build()
    lib = capi.load()
    fake = ctypes.c_void_p(0x1000)
    p = capi.VerifyParams().to_c()
    B, K, V = 4096, 4, 262144
    assert lib.spec_verify_workspace_bytes(B, K, V) > 16 << 20
    rc = lib.spec_verify_noalloc(fake, 1, B, K, V, fake, None, fake, None, 0, None, ctypes.byref(p),
                                 fake, fake, fake, fake, None)
    assert rc == -5                                           # SPECNG_ESMALL
    msg = lib.specng_last_error()
    assert b"B=4096" in msg and b"static scratch" in msg
    assert lib.spec_verify_workspace_bytes(512, 4, 262144) <= 16 << 20
    rc = lib.spec_verify_noalloc(fake, 1, 0, K, V, fake, None, fake, None, 0, None, ctypes.byref(p),
                                 fake, fake, fake, fake, None)
    assert rc == -1
