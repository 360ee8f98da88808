"""Pins for the oracle's Philox4x32-10 and its uniform / Gumbel maps.

The oracle's generator is checked against an implementation it shares no
code with: Triton's ``tl.random.philox`` (the published Philox4x32-10 of
Salmon et al., SC'11), run by Triton's CPU interpreter in a subprocess.
"""
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
from scipy import stats

from oracle import philox

_TRITON_SCRIPT = textwrap.dedent(r"""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def kern(c_ptr, o_ptr, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        c0 = tl.load(c_ptr + i * 4 + 0).to(tl.uint32, bitcast=True)
        c1 = tl.load(c_ptr + i * 4 + 1).to(tl.uint32, bitcast=True)
        c2 = tl.load(c_ptr + i * 4 + 2).to(tl.uint32, bitcast=True)
        c3 = tl.load(c_ptr + i * 4 + 3).to(tl.uint32, bitcast=True)
        a, b, c, d = tl.random.philox(seed, c0, c1, c2, c3)
        tl.store(o_ptr + i * 4 + 0, a.to(tl.int32, bitcast=True))
        tl.store(o_ptr + i * 4 + 1, b.to(tl.int32, bitcast=True))
        tl.store(o_ptr + i * 4 + 2, c.to(tl.int32, bitcast=True))
        tl.store(o_ptr + i * 4 + 3, d.to(tl.int32, bitcast=True))

    spec = json.loads(sys.stdin.read())
    ctr = np.array(spec["ctr"], dtype=np.uint32).view(np.int32)
    out = torch.zeros(ctr.size, dtype=torch.int32)
    kern[(1,)](torch.from_numpy(ctr.copy()), out, spec["seed"], N=ctr.size // 4)
    print(json.dumps(out.numpy().view(np.uint32).tolist()))
""")


def _triton_philox(ctr: np.ndarray, seed: int) -> np.ndarray:
    pytest.importorskip("triton")
    env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT],
                         input=json.dumps({"ctr": ctr.reshape(-1).tolist(), "seed": int(seed)}),
                         capture_output=True, text=True, env=env, timeout=600)
    if res.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + res.stderr.strip().splitlines()[-1])
    return np.array(json.loads(res.stdout.strip().splitlines()[-1]), dtype=np.uint64).reshape(-1, 4)


@pytest.mark.parametrize("seed", [0, 0x0123456789ABCDEF, (1 << 64) - 1])
def test_philox_matches_independent_implementation(seed):
    rng = np.random.default_rng(11)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    ctr[1] = 0xFFFFFFFF
    ref = _triton_philox(ctr, seed)
    k0, k1 = philox.seed_key(seed)
    got = np.stack(philox.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], k0, k1), axis=1)
    np.testing.assert_array_equal(got, ref)


def test_philox_is_not_identity_and_depends_on_every_input():
    base = np.array(philox.philox4x32_10(1, 2, 3, 4, 5, 6))
    for change in [(2, 2, 3, 4, 5, 6), (1, 3, 3, 4, 5, 6), (1, 2, 4, 4, 5, 6),
                   (1, 2, 3, 5, 5, 6), (1, 2, 3, 4, 6, 6), (1, 2, 3, 4, 5, 7)]:
        other = np.array(philox.philox4x32_10(*change))
        assert (other != base).all()


def test_uniform_grid_is_exact_and_open():
    w = np.array([0, 511, 512, 2**32 - 1, 2**31], dtype=np.uint64)
    u = philox.uniform_from_word(w)
    assert u[0] == 2.0 ** -24 and u[1] == 2.0 ** -24
    assert u[2] == 3 * 2.0 ** -24
    assert u[3] == 1.0 - 2.0 ** -24
    assert u[4] == 0.5 + 2.0 ** -24
    assert np.all(u.astype(np.float32).astype(np.float64) == u)   # exact in fp32
    assert np.all((u > 0) & (u < 1))


def test_gumbel_map_closed_form_and_range():
    u = np.array([np.exp(-1.0), 0.5, 1 - 2.0 ** -24, 2.0 ** -24])
    g = philox.gumbel_from_uniform(u)
    assert abs(g[0] - 0.0) < 1e-15                     # -ln(-ln e^-1) = 0
    assert abs(g[1] + np.log(np.log(2.0))) < 1e-15
    assert 16.6 < g[2] < 16.7 and -2.82 < g[3] < -2.80
    # the upper tail uses log1p(u - 1): compare with a long-double reference
    uu = 1 - np.arange(1, 1000) * 2.0 ** -24
    ref = -np.log(-np.log1p(np.longdouble(uu) - 1))
    np.testing.assert_allclose(philox.gumbel_from_uniform(uu), ref.astype(np.float64), rtol=0, atol=1e-13)


def test_uniformity_chisq():
    seq = np.arange(4096)
    u = philox.accept_uniform(123, seq, 9, 1)
    g_words = philox.gumbel_noise(123, 3, 9, 0, np.arange(200000))
    for sample in (u, np.exp(-np.exp(-g_words))):
        counts, _ = np.histogram(sample, bins=64, range=(0, 1))
        p = stats.chisquare(counts).pvalue
        assert p > 1e-4, p


def test_counter_layout_lanes():
    # four consecutive vocab ids share one Philox block for their element draws and take its four
    # words; 256 consecutive ids share one block draw (M = E(word 0) / 256, I = word 1 & 255)
    k0, k1 = philox.seed_key(77)
    words = philox.philox4x32_10(5, 3, 8, 2, k0, k1)
    F = philox.exp_from_uniform(philox.uniform_from_word(np.array([int(w) for w in words], dtype=np.uint64)))
    b0, b1, _, _ = philox.philox4x32_10(0, 3 | (2 << 16), 8, 2, k0, k1)
    M = philox.exp_from_uniform(philox.uniform_from_word(np.uint64(int(b0)))) / 256
    I = int(b1) & 255
    ids = np.arange(20, 24)
    E = np.where(ids == I, M, M + F)
    np.testing.assert_array_equal(philox.exp_noise(77, 2, 8, 3, ids), E)
    np.testing.assert_array_equal(philox.gumbel_noise(77, 2, 8, 3, ids), -np.log(E))
    # the id at the block's argmin slot carries M alone
    assert philox.exp_noise(77, 2, 8, 3, I) == M
    ua = philox.accept_uniform(77, 2, 8, 3)
    w0 = philox.philox4x32_10(0, 3 | (1 << 16), 8, 2, k0, k1)[0]
    assert ua == philox.uniform_from_word(w0)


def test_gumbel_row_equals_per_id_noise():
    seq = np.array([0, 5, 9])
    pos = np.array([0, 2, 4])
    for V in (1, 7, 8, 33, 256, 1100):
        row = philox.gumbel_row(3, seq, 11, pos, V)
        ref = philox.gumbel_noise(3, seq[:, None], 11, pos[:, None], np.arange(V)[None, :])
        np.testing.assert_array_equal(row, ref)
        np.testing.assert_array_equal(philox.exp_row(3, seq, 11, pos, V),
                                      philox.exp_noise(3, seq[:, None], 11, pos[:, None], np.arange(V)[None, :]))


def test_exp_map_closed_form():
    u = np.array([np.exp(-1.0), 0.5, 1 - 2.0 ** -24, 2.0 ** -24])
    E = philox.exp_from_uniform(u)
    assert abs(E[0] - 1.0) < 1e-15 and abs(E[1] - np.log(2.0)) < 1e-16
    assert E[2] == -np.log1p(-2.0 ** -24) and abs(E[3] - 24 * np.log(2.0)) < 1e-13


NB = philox.NOISE_BLOCK


def _block_rows(n, V=2 * NB, seed=2718, step=5, pos=1):
    return philox.exp_row(seed, np.arange(n), step, pos, V)


def _block_law_pvalues(E):
    """p-values of the order-statistics laws of the first two blocks of rows
    E [n, >= 2 NB] and of the Exp(1) marginals of a few ids."""
    n = E.shape[0]
    pv = []
    for blk in (0, 1):
        sl = E[:, blk * NB:(blk + 1) * NB]
        e = np.sort(sl, axis=1)
        pv.append(stats.kstest(NB * e[:, 0], "expon").pvalue)                # minimum ~ Exp(NB)
        pv.append(stats.kstest((NB - 1) * (e[:, 1] - e[:, 0]), "expon").pvalue)  # next gap ~ Exp(NB - 1)
        counts = np.bincount(np.argmin(sl, axis=1) * 64 // NB, minlength=64)  # argmin uniform
        pv.append(stats.chisquare(counts).pvalue)
    for v in (0, 1, NB // 2 - 1, NB - 1, NB, 2 * NB - 1):
        pv.append(stats.kstest(E[:, v], "expon").pvalue)
    c = np.corrcoef(E[:, [0, 1, NB // 2 + 5, NB - 1, NB]].T)
    pv.append(1.0 if np.abs(c[~np.eye(5, dtype=bool)]).max() < 5 / np.sqrt(n) else 0.0)
    return np.array(pv)


def test_block_construction_laws():
    """The block draw must leave the E_v of a block i.i.d. Exp(1).  Order
    statistics of n i.i.d. Exp(1) (Renyi): the minimum is Exp(n), the gap to
    the second smallest is Exp(n - 1), the argmin is uniform; and every
    marginal is Exp(1) with no correlation between ids."""
    assert _block_law_pvalues(_block_rows(6000)).min() > 1e-3


@pytest.mark.parametrize("mistake", ["no_min_added", "argmin_on_half", "min_rate_1", "no_argmin_slot"])
def test_block_pins_catch_planted_mistakes(mistake):
    """Each plausible slip in the block construction, planted in a copy built
    from the oracle's own draws, fails the law checks above."""
    n, V = 3000, 2 * NB
    seq = np.arange(n)[:, None]
    v = np.arange(V)[None, :]
    M, I = philox.block_draw(11, seq, 3, 0, v // NB)
    F = philox.element_exp(11, seq, 3, 0, v)
    slot = v % NB
    if mistake == "no_min_added":
        E = np.where(slot == I, M, F)
    elif mistake == "argmin_on_half":
        E = np.where(slot == (I % (NB // 2)), M, M + F)
    elif mistake == "min_rate_1":
        E = np.where(slot == I, M * NB, M * NB + F)
    else:
        E = M + F
    assert _block_law_pvalues(E).min() < 1e-6
    # the unmodified composition of the same draws passes
    if mistake == "no_argmin_slot":
        assert _block_law_pvalues(np.where(slot == I, M, M + F)).min() > 1e-3


def test_gumbel_max_over_blocks_matches_softmax():
    """argmax_v (log p_v - ln E_v) is distributed as p, with the mass spread
    across the boundary of two blocks."""
    V = 4 * NB
    v = np.arange(V)
    x = -np.abs(v - (2 * NB - 0.5)) / 3.0
    logp = x - (x.max() + np.log(np.sum(np.exp(x - x.max()))))
    n = 20000
    g = -np.log(_block_rows(n, V, seed=99, step=1, pos=0))
    y = np.argmax(logp[None, :] + g, axis=1)
    counts = np.bincount(y, minlength=V).astype(float)
    exp = np.exp(logp) * n
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    assert stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue > 1e-3
