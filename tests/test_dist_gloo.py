"""The bench's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank runs its own replica (weak scaling, no collective on the data path)
or, with --shard, a contiguous range of one model's blocks (strong scaling);
the only collectives are the barrier around the timed region, the max of the
ranks' times and the sum of their parameter counts. Also checks that the
replicas draw disjoint state and that the shards cover the model.
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


def _shard_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    bench.dist_init("gloo")
    L, first = bench.rank_layout("tinyllama_full_l16m", 0, True, rank, world)
    total = bench.sum_over_ranks(L.n_params)
    got = [None] * world
    dist.all_gather_object(got, (first, L.n_layers, L.n_params))
    q.put((rank, total, got))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_one_model():
    """--shard: the ranks' block ranges are contiguous, disjoint and cover the
    model; the job's parameter count (the sum over ranks) is the model's."""
    import bench
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    full = bench.build_layout("tinyllama_full_l16m")
    for (_, total, got) in res:
        assert total == full.n_params
        (f0, n0, p0), (f1, n1, p1) = got
        assert f0 == 0 and f1 == n0 and n0 + n1 == full.n_layers and p0 + p1 == full.n_params


def test_shard_blocks_cover_and_balance():
    import bench
    sizes = [1_000] + [700] * 22 + [1_000]
    for world in (1, 2, 3, 4, 8, 24):
        r = bench.shard_blocks(sizes, world)
        assert len(r) == world and r[0][0] == 0 and r[-1][1] == len(sizes)
        assert all(a < b for a, b in r)  # every rank has a block
        assert all(r[k][1] == r[k + 1][0] for k in range(world - 1))  # contiguous, disjoint
        loads = [sum(sizes[a:b]) for a, b in r]
        assert max(loads) - min(loads) <= 2 * max(sizes)  # balanced to within two blocks
    r = bench.shard_blocks([5, 5], 4)  # fewer blocks than ranks: some ranges empty
    assert r[0][0] == 0 and r[-1][1] == 2 and sum(b - a for a, b in r) == 2
    assert bench.shard_blocks([3, 1, 1, 1], 2) == [(0, 1), (1, 4)]


def test_single_process_defaults():
    import bench
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 0, 1)
    assert bench.max_over_ranks(3.25) == 3.25


def test_replicas_fit_host_memory():
    """The bench's guard for one pinned replica of the state per rank: the
    state plus the health check's allowance, times the ranks on the host,
    within 3/4 of the available memory; an unknown availability does not
    block."""
    import bench
    GB = 1 << 30
    state = 82 * GB   # the Llama-70B slice
    assert bench.replicas_fit(state, 1, 200 * GB)          # one GPU on a ~200 GB host
    assert not bench.replicas_fit(state, 2, 200 * GB)
    assert bench.replicas_fit(state, 8, 1600 * GB)         # 8 x (82 + 40) = 976 GB
    assert not bench.replicas_fit(state, 8, 1000 * GB)
    assert bench.replicas_fit(state, 8, 0)
    assert bench.replicas_fit(GB, 8, 64 * GB)              # small states: half the state as allowance
    assert bench.host_mem_available() >= 0
