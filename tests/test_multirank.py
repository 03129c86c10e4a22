"""The multi-rank host logic of bench.py on CPU: two gloo ranks (world_size 2).

Under torchrun every rank scores its own problems (no data-path collective); the only
communication is the barrier around the timed region and the max-reduction of the
elapsed time.  Checked here without a GPU: the ranks' workloads differ, every rank
gets the slowest rank's time, and a rank that fails raises on the host."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    w = bench.rank_workload(synth.WORKLOADS["c3"], rank)
    keys = synth.unit_keys(w.seed, 0, 0, 4, w.D)
    elapsed = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    dist.barrier()
    slowest = bench.max_over_ranks(elapsed, dist, "cpu")
    out[rank] = (w.seed, float(keys[0, 0]), slowest)
    dist.destroy_process_group()


def test_two_gloo_ranks_partition_and_max():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for pr in procs:
            pr.start()
        for pr in procs:
            pr.join(120)
            assert pr.exitcode == 0
        (s0, k0, m0), (s1, k1, m1) = out[0], out[1]
    assert s0 != s1 and k0 != k1                     # each rank its own problems
    assert m0 == m1 == 15.0                          # both see the slowest rank's time


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
