"""Host-side helpers of bench.py (no GPU)."""
import torch

import bench


def test_step_summary_counts_accept_lengths_and_tokens():
    # two steps, three sequences, K = 4
    acc = torch.tensor([[0, 2, 4], [1, 0, 3]], dtype=torch.int32)
    k = torch.tensor([[4, 2, 4], [3, 0, 4]], dtype=torch.int32)
    m = bench.step_summary(acc, k, 4)
    assert m["steps"] == 2
    assert m["accept_len_hist"] == [2, 1, 1, 1, 1]
    assert m["tokens_per_sequence_step"] == (1 + 3 + 5 + 2 + 1 + 4) / 6
    assert m["tokens_per_step"] == ((1 + 3 + 5) + (2 + 1 + 4)) / 2
    assert m["drafts_offered_per_step"] == (10 + 7) / 2
    assert m["acceptance_rate"] == (0 + 2 + 4 + 1 + 0 + 3) / 17


def test_step_summary_without_drafts():
    acc = torch.zeros((3, 2), dtype=torch.int32)
    k = torch.zeros((3, 2), dtype=torch.int32)
    m = bench.step_summary(acc, k, 2)
    assert m["accept_len_hist"] == [6, 0, 0]
    assert m["acceptance_rate"] is None
    assert m["tokens_per_step"] == 2.0
