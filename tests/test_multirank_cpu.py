"""The multi-rank host logic of the benchmark on CPU with the gloo backend (world
size 2): every rank gets its own sequences (no data-path collective), and the
step time reported is the maximum over ranks."""
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


def _worker(rank, world, port, B, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from sparse_depth_token_gb300 import inputs as I
    # sequences owned by this rank, as a strong-scaling split of B sequences
    mine = list(I.shard_sequences(B, rank, world))
    got = [None] * world
    dist.all_gather_object(got, mine)
    # per-rank data under weak scaling: the benchmark offsets the seed by rank
    w = I.WORKLOADS["tiny_fp32"]
    wr = w.replace(seed=w.seed + 1000 * rank) if rank else w
    x = torch.from_numpy(I.residual_stream(wr)[0, 0, :4].copy())
    xs = [torch.zeros(4) for _ in range(world)]
    dist.all_gather(xs, x)
    # max-over-ranks of the step time
    t = torch.tensor([10.0 + rank])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        out.put((got, [v.tolist() for v in xs], float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, 7, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, xs, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got[0] + got[1] == list(range(7))           # disjoint, complete, in order
    assert abs(len(got[0]) - len(got[1])) <= 1
    assert xs[0] != xs[1]                              # each rank runs its own sequences
    assert tmax == 11.0


def test_shard_sequences_properties():
    from sparse_depth_token_gb300 import inputs as I
    for B in (1, 4, 7, 64):
        for world in (1, 2, 3, 8):
            parts = [list(I.shard_sequences(B, r, world)) for r in range(world)]
            assert sum(parts, []) == list(range(B))
            assert max(map(len, parts)) - min(map(len, parts)) <= 1
