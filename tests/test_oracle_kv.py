"""Pins of the KV block pool oracle (CPU): hand-worked traces, conservation,
closed forms."""
import random

from oracle import kv as ok


def test_blocks_for_closed_form():
    assert [ok.blocks_for(n, 4) for n in (-3, 0, 1, 4, 5, 8, 9)] == [0, 0, 1, 1, 2, 2, 3]
    assert ok.blocks_for(16, 16) == 1 and ok.blocks_for(17, 16) == 2


def test_hand_worked_trace_one_sequence():
    # block_size 4, 6 blocks.  A forward of 5 positions from kv_len 0 needs 2
    # blocks (0 and 1); rollback to kv_len 3 keeps block 0 and returns block 1;
    # the next forward of 5 from 3 needs ceil(8 / 4) = 2 blocks: block 1 again.
    p = ok.KvPool(6, 1, 8, 4)
    p.reserve([0], 5)
    assert p.tables == [[0, 1]] and p.free == [5, 4, 3, 2]
    p.trim([3])
    assert p.tables == [[0]] and p.free == [5, 4, 3, 2, 1]
    p.reserve([3], 5)
    assert p.tables == [[0, 1]]
    p.release([1])
    assert p.tables == [[]] and sorted(p.free) == list(range(6)) and not p.short


def test_hand_worked_trace_two_sequences_short():
    # 3 blocks of 2 positions: sequence 0 wants ceil(3 / 2) = 2, sequence 1
    # wants ceil(4 / 2) = 2, only one is left for it: short
    p = ok.KvPool(3, 2, 4, 2)
    p.reserve([1, 2], 2)
    assert p.tables == [[0, 1], [2]] and p.short and p.free == []


def test_table_row_cap_is_short():
    p = ok.KvPool(10, 1, 2, 4)
    p.reserve([0], 12)  # wants 3, the row holds 2
    assert p.counts() == [2] and p.short


def test_conservation_random_traces():
    rng = random.Random(5)
    for _ in range(200):
        nb, B, mb, bs = rng.randint(1, 40), rng.randint(1, 6), rng.randint(1, 8), rng.randint(1, 5)
        p = ok.KvPool(nb, B, mb, bs)
        kv = [rng.randint(0, 10) for _ in range(B)]
        for _ in range(10):
            op = rng.random()
            if op < 0.5:
                p.reserve(kv, rng.randint(0, 5))
            elif op < 0.8:
                kv = [max(0, x - rng.randint(0, 4)) for x in kv]
                p.trim(kv)
            else:
                p.release([rng.random() < 0.3 for _ in range(B)])
            held = [blk for t in p.tables for blk in t]
            assert sorted(held + p.free) == list(range(nb))          # every block exactly once
            for b in range(B):
                assert len(p.tables[b]) <= mb
