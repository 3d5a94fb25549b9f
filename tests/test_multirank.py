"""World-size-2 checks of the data-parallel split on CPU (gloo): whole sequences are
sharded across ranks, each rank computes its shard alone (here with the CPU oracle), and
the union of the shards equals the single-process result; the timing reduction takes the
slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from mamba2_ssd_state_gb300 import shard

SEQS = [40, 7, 0, 23, 16, 31, 2]


def test_partition_sequences_balances_and_covers():
    parts = shard.partition_sequences([8192, 3000, 517, 4675], 2)
    assert sorted(sum(parts, [])) == [0, 1, 2, 3]
    loads = [sum([8192, 3000, 517, 4675][i] for i in p) for p in parts]
    assert max(loads) - min(loads) <= 8192
    assert shard.partition_sequences([5], 3) == [[0], [], []]
    assert shard.partition_rows(7, 3) == [[0, 1, 2], [3, 4], [5, 6]]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from mamba2_ssd_state_gb300 import inputs as I

        s = I.make_scan_inputs(SEQS, H=2, P=4, G=1, N=8, chunk_size=8, act="f32", seed=5,
                               init=[1, 0, 1, 0, 1, 1, 0])
        mine = shard.partition_sequences(SEQS, world)[rank]
        out = {}
        for i in mine:  # each sequence is independent: run it on its own
            a, b = int(s.cu_seqlens[i]), int(s.cu_seqlens[i + 1])
            y, fin = oracle.scan_seq(s.x.values[a:b], s.dt.values[a:b], s.A.values,
                                     s.B.values[a:b], s.C.values[a:b], D=s.D.values,
                                     dt_bias=s.dt_bias.values,
                                     initial_states=s.initial_states.values[i:i + 1],
                                     has_initial_state=s.has_initial_state[i:i + 1])
            out[i] = (y, fin[0])
        gathered = [None] * world
        dist.all_gather_object(gathered, out)   # test-side check only
        slowest = shard.max_over_ranks(10.0 + rank)
        if rank == 0:
            q.put((gathered, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_equal_single_process():
    import oracle
    from mamba2_ssd_state_gb300 import inputs as I

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, slowest = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert slowest == 11.0
    s = I.make_scan_inputs(SEQS, H=2, P=4, G=1, N=8, chunk_size=8, act="f32", seed=5,
                           init=[1, 0, 1, 0, 1, 1, 0])
    y, fin = oracle.scan_seq(s.x.values, s.dt.values, s.A.values, s.B.values, s.C.values,
                             D=s.D.values, dt_bias=s.dt_bias.values,
                             initial_states=s.initial_states.values,
                             has_initial_state=s.has_initial_state, cu_seqlens=s.cu_seqlens)
    merged = {}
    for part in gathered:
        merged.update(part)
    assert sorted(merged) == list(range(len(SEQS)))
    for i, (yi, fi) in merged.items():
        a, b = int(s.cu_seqlens[i]), int(s.cu_seqlens[i + 1])
        np.testing.assert_allclose(yi, y[a:b], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(fi, fin[i], rtol=1e-13, atol=1e-14)
