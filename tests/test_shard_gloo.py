"""Multi-rank path on CPU: two gloo ranks each take their shard of a global
batch, compute it (with the oracle, standing in for the GPU kernels), and the
gathered shards must equal the whole; the max-over-ranks timing reduction is
the one bench.py uses."""
import os
import socket

import numpy as np
import pytest

from alibi_positional_bias_gb300.shard import shard_batch, shard_range


def test_shard_range_covers_everything():
    for units in (0, 1, 5, 64, 2560):
        for world in (1, 2, 3, 8):
            parts = [shard_range(units, world, r) for r in range(world)]
            assert sum(c for _, c in parts) == units
            pos = 0
            for s, c in parts:
                assert s == pos
                pos += c
            counts = [c for _, c in parts]
            assert max(counts) - min(counts) <= 1
    with pytest.raises(ValueError):
        shard_range(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import alibi_inputs as gen
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = gen.Workload("gloo", "prefill", 3, 2, 40, 16, "bf16", seed=5)
        q_, k_, v_ = gen.generate(w)
        b0, nb = shard_batch(w.B, world, rank)
        out, lse, _ = oracle.attention(q_.f32[b0:b0 + nb], k_.f32[b0:b0 + nb], v_.f32[b0:b0 + nb], nthreads=1)
        mine = torch.from_numpy(np.ascontiguousarray(out.reshape(nb, -1)))
        gathered = [None] * world
        dist.all_gather_object(gathered, (b0, nb, mine.numpy()))
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            full, _, _ = oracle.attention(q_.f32, k_.f32, v_.f32, nthreads=1)
            got = np.zeros_like(full.reshape(w.B, -1))
            for s, c, arr in gathered:
                got[s:s + c] = arr
            q.put((bool(np.array_equal(got, full.reshape(w.B, -1))), float(t[0])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_whole():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    equal, tmax = q.get(timeout=10)
    assert equal and tmax == 2.0
