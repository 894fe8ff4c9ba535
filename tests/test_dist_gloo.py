"""The bench's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank runs its own replica (weak scaling, no collective on the data path);
the only collectives are the barrier around the timed region and the max of
the ranks' times. Also checks that the replicas draw disjoint state.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import bench
    import synth
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world) and bench.dist_env() == (rank, rank, world)
    bench.barrier()
    t = bench.max_over_ranks(1.5 + rank)
    seed = bench.replica_seed(0x5EED, rank)
    a = np.empty(64, np.float32)
    synth.fill(a, synth.KIND_F32, seed, synth.stream_id(synth.FIELD_G, 0), 0, 1e-3)
    got = [None] * world
    dist.all_gather_object(got, a.tobytes())
    q.put((rank, t, got[0] != got[1]))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_disjoint_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert [r for (r, _, _) in res] == [0, 1]
    assert all(t == 2.5 for (_, t, _) in res)  # max over ranks
    assert all(d for (_, _, d) in res)  # replicas draw different state


def test_single_process_defaults():
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(3.25) == 3.25
