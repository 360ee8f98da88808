"""The N > 1 host logic of bench.py, on CPU with gloo (world size 2): each
rank gets the same shapes with its own seeds (weak scaling, no collective on
the data path), the timed region is reduced by a max over ranks, and the
reference arm runs on rank 0 only."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from speculative_decoding_draft_ngram_gb300 import workloads as wl
    res = {}
    res["max"] = bench.max_over_ranks(10.0 + rank, "cpu")
    cfg = bench.rank_config("c5", 50, rank, batch=4)
    res["shape"] = (cfg.B, cfg.K, cfg.V, cfg.steps)
    res["seeds"] = (cfg.data_seed, cfg.sampler_seed)
    small = wl.get("c1", data_seed=cfg.data_seed)
    hist, lens = wl.histories(small, "cpu")
    res["hist_sum"] = int(hist[:, :64].sum())

    class Args:
        workload = "c5"
        cpu_sample = 1
        warmup = 0
        steps = 0
    # the reference arm: rank 0 alone does work; the other ranks return at once
    res["ref_returned"] = bench.run_reference(Args()) is None if rank != 0 else True
    gathered = [None] * world
    dist.all_gather_object(gathered, res)
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = q.get(timeout=300)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    r0, r1 = got
    assert r0["max"] == r1["max"] == 11.0
    assert r0["shape"] == r1["shape"] == (4, 4, 151936, 200)
    assert r0["seeds"] != r1["seeds"]
    assert r0["hist_sum"] != r1["hist_sum"]
    assert r1["ref_returned"]
