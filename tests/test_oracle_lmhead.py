"""Pins of oracle/lmhead.py (CPU)."""
import numpy as np
import torch

from oracle import lmhead as ol


def test_dot_products_hand_worked():
    h = np.array([[1.0, 2.0, 3.0], [-1.0, 0.0, 2.0]])
    w = np.array([[1.0, 1.0, 1.0], [2.0, -1.0, 0.0]])
    # [1+2+3, 2-2+0], [-1+0+2, -2+0+0]
    np.testing.assert_array_equal(ol.lm_head_logits(h, w), [[6.0, 0.0], [1.0, -2.0]])


def test_against_a_triple_loop():
    rng = np.random.default_rng(3)
    h = rng.integers(-3, 4, size=(2, 3, 17)).astype(np.float64) / 8
    w = rng.integers(-3, 4, size=(11, 17)).astype(np.float64) / 8
    got = ol.lm_head_logits(h, w)
    for b in range(2):
        for j in range(3):
            for v in range(11):
                s = 0.0
                for i in range(17):
                    s += h[b, j, i] * w[v, i]
                assert got[b, j, v] == ol.bf16_round(s)


def test_rounding_ties_go_to_even():
    cases = {
        257.0: 256.0,             # spacing 2 in [256, 512): a tie, 256 has the even significand
        259.0: 260.0,             # tie between 258 (odd) and 260 (even)
        1.0 + 2.0 ** -8: 1.0,     # tie at the 8th bit
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,
        -300.5: -300.0,           # nearest, not a tie
        1.5: 1.5,
        0.0: 0.0,
        -(2.0 ** -126): -(2.0 ** -126),
    }
    for x, y in cases.items():
        assert ol.bf16_round(np.float64(x)) == y, x


def test_rounding_matches_torch_conversion():
    # fp32 values (exact in fp64) rounded by torch's own fp32 -> bf16 conversion
    g = torch.Generator().manual_seed(0)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-20, 20, (20000,), generator=g).float())
    ref = x.to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ol.bf16_round(x.double().numpy()), ref)
