"""Multi-process host logic on CPU (gloo, world size 2): the scalar all-reduce
of the shard statistics gives every rank bit-identical totals equal to the
oracle's rank-order fold; shard bounds partition the buffer across processes;
the benchmark's max-over-ranks timing.  No GPU is touched."""
import os
import socket

import numpy as np
import pytest

from conftest import spawn_bounded

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUMEL = 100_003


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_grads(r, world, inject):
    import oracle as O
    import synth
    b, e, _, _ = O.shard_bounds(NUMEL, world, r)
    bufs = [synth.normal_np(17, 1 + i, b, e - b, 3.0, synth.F16) for i in range(2)]
    if r == 1 and inject:
        bufs[0][5] = 0x7C00
    return bufs


def _worker(rank, world, port, out_dir, inject):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    import bench
    import oracle as O
    import zero_sharded_mixed_05_gb300 as z
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    h = z.zero_opt_create(z.make_config(numel=NUMEL, world=world))
    b, e, S, P = z.zero_opt_shard_bounds(h, rank)
    assert (b, e, S, P) == O.shard_bounds(NUMEL, world, rank)
    own = O.stats_of(O.reduce(_shard_grads(rank, world, inject), O.FP16))
    G = z.allgather_fold(z.zero_opt_stats(own.sumsq, own.nonfinite, 0))
    t = bench.max_over_ranks(1.5 + rank, "cpu")
    np.save(os.path.join(out_dir, f"r{rank}.npy"),
            np.array([G.sumsq, G.nonfinite, t, b, e], dtype=np.float64))
    z.zero_opt_destroy(h)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("inject", [False, True])
def test_two_rank_stats_exchange(tmp_path, inject):
    from zero_sharded_mixed_05_gb300 import _build
    _build.build()
    import oracle as O
    world = 2
    spawn_bounded(_worker, (world, _free_port(), str(tmp_path), inject), world)
    rows = [np.load(os.path.join(tmp_path, f"r{r}.npy")) for r in range(world)]
    assert rows[0][0].tobytes() == rows[1][0].tobytes()        # identical bits
    assert rows[0][1] == rows[1][1] == float(inject)
    ref = O.fold_stats([O.stats_of(O.reduce(_shard_grads(r, world, inject), O.FP16))
                        for r in range(world)])
    if not inject:
        assert rows[0][0] == ref.sumsq
    assert ref.nonfinite == int(inject)
    assert rows[0][2] == rows[1][2] == 2.5                       # max over ranks
    assert rows[0][3] == 0 and rows[0][4] == rows[1][3] and rows[1][4] == NUMEL
