"""Multi-rank glue of bench.py on CPU (gloo, world size 2).

bench.py runs one independent replica per GPU (weak scaling): no data-path
collective, only a barrier and max-over-ranks time / sum-over-ranks units.
These tests run that glue in two spawned CPU processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    w, r, lr = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    # each rank reports its own time and units; the job time is the slowest rank
    t = bench.max_over_ranks(1.0 + rank, dist)
    u = bench.sum_over_ranks(100.0 * (rank + 1), dist)
    wl = bench.rank_workload("tiny", rank)
    out[rank] = (w, r, lr, t, u, wl.seed_logits, wl.seed_x)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_glue():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    r0, r1 = out[0], out[1]
    assert r0[:3] == (2, 0, 0) and r1[:3] == (2, 1, 1)
    assert r0[3] == r1[3] == 2.0            # max over ranks
    assert r0[4] == r1[4] == 300.0          # units of all ranks
    assert r0[5] != r1[5] and r0[6] != r1[6]  # each rank draws its own batch


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.sum_over_ranks(7.0, None) == 7.0


@pytest.mark.parametrize("name", ["tiny", "prefill"])
def test_byte_model_matches_hand_count(name):
    sys.path.insert(0, ROOT)
    import bench
    import moe_synth as ms
    w = ms.workload(name)
    c, pairs = 3 * w.T, w.T * w.k
    b = bench.algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, c, c, pairs)
    row = w.H * 2
    assert b["pack"] == w.T * row + c * row + c * 4
    assert b["permute"] == c * row + pairs * row + w.T * w.k * 8
    assert b["combine"] == pairs * row + w.T * w.k * 8 + w.T * row
    assert b["step"] == b["route"] + b["layout"] + b["pack"] + b["permute"] + b["combine"]
