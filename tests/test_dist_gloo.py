"""Data-parallel synchronisation of the block moments, on CPU ranks (gloo).

Each data-parallel replica accumulates its own EMA of block moments; before a
refresh the replicas average their A buffers with one all-reduce ("Dobb",
Abstract: "no communication beyond data-parallel synchronization of the
activation second moments"; Table 3 caption: n^2/B entries per matrix).
Because the EMA is linear, replacing every replica's A by the average at
refresh time gives exactly the EMA of the averaged moments, at every later
refresh as well.  The test runs two processes with the oracle's arithmetic
and the same all-reduce the benchmark issues for N > 1 GPUs."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import dobb as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    n, B, beta2, T, steps = 12, 3, 0.9, 3, 7
    k = n // B
    rng = np.random.default_rng(100)  # the same stream on every rank
    streams = [[rng.standard_normal((9, n)) for _ in range(steps)] for _ in range(world)]
    A = np.zeros((B, k, k))
    synced = []
    for t in range(steps):
        A = O.block_moment_ema(A, streams[rank][t], beta2, B)
        if t % T == 0:
            buf = torch.from_numpy(A.copy())
            dist.all_reduce(buf, op=dist.ReduceOp.SUM)
            A = (buf / world).numpy()
            synced.append(A.copy())
    # reference: EMA of the averaged per-step moments
    Aref = np.zeros((B, k, k))
    refs = []
    for t in range(steps):
        mom = sum(O.block_moment_ema(np.zeros((B, k, k)), streams[r][t], 0.0, B)
                  for r in range(world)) / world
        Aref = beta2 * Aref + (1 - beta2) * mom
        if t % T == 0:
            refs.append(Aref.copy())
    err = max(float(np.abs(a - b).max()) for a, b in zip(synced, refs))
    out_q.put((rank, err, len(synced)))
    dist.barrier()
    dist.destroy_process_group()


def test_moment_allreduce_equals_ema_of_averaged_moments():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, n_sync in res:
        assert n_sync == 3
        assert err < 1e-13


def _placement_worker(rank, world, port, out_q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    from block_eigenbasis_preconditioning_gb300.sharding import matrix_cost, partition_matrices
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shapes = I.gpt2_xl_shapes().shapes
    owned = partition_matrices(shapes, 16, world)
    mine = torch.tensor(owned[rank] + [-1] * (len(shapes) - len(owned[rank])), dtype=torch.int64)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    lists = [[int(v) for v in g.tolist() if v >= 0] for g in gathered]
    cost = [sum(matrix_cost(*shapes[i], 16, 8192, 10) for i in lst) for lst in lists]
    out_q.put((rank, lists == owned, sorted(sum(lists, [])) == list(range(len(shapes))),
               max(cost) / min(cost)))
    dist.barrier()
    dist.destroy_process_group()


def test_matrix_placement_across_ranks():
    """Two ranks compute the placement of the GPT-2 XL matrices on their own
    and agree on it (exchanged with an all-gather); every matrix is owned by
    exactly one rank and the estimated loads differ by less than 5 %."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_placement_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, cover, imbalance in res:
        assert same and cover
        assert imbalance < 1.05
