"""Plan A among CPU ranks (gloo, world sizes 2 and 3): each rank builds its
schedule with the library's host planner, packs its rows in
destination-local order, runs the variable-split all_to_all_single that the
split sizes define, and reorders what it receives with recv_index.  Every
rank must end with exactly its destination rows.  That is the single-rank
transition restricted to the rank ("Window-Aligned Sequence Parallelism
(SeedVR2)", section "Plan A redistribution").  On CPU the pack and unpack
gathers are torch indexing on the same index tables the device gather uses."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

GRID = (7, 24, 40, 3, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, layouts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import shifted_window_attention_gb300.sp as sp
        src_l, dst_l = layouts
        N = GRID[0] * GRID[1] * GRID[2]
        x = torch.arange(N, dtype=torch.float64)[:, None] * torch.tensor([[1.0, -1.0, 0.5]])  # canonical rows
        rows = sp.local_rows(*GRID, src_l, world, rank)
        x_local = x[torch.from_numpy(rows.astype(np.int64))]
        pa = sp.PlanA(*GRID, src_l, dst_l, world, rank)
        flags = [None] * world
        dist.all_gather_object(flags, pa.network_exchange_required)
        if pa.network_exchange_required:
            send = x_local[torch.from_numpy(pa.send_index.astype(np.int64))]
            recv = torch.empty((pa.n_recv, 3), dtype=torch.float64)
            dist.all_to_all_single(recv, send, output_split_sizes=pa.output_split_sizes,
                                   input_split_sizes=pa.input_split_sizes)
            y = recv[torch.from_numpy(pa.recv_index.astype(np.int64))]
        else:
            y = x_local[torch.from_numpy(pa.send_index[pa.recv_index].astype(np.int64))]
        want = x[torch.from_numpy(sp.local_rows(*GRID, dst_l, world, rank).astype(np.int64))]
        out[rank] = (bool(torch.equal(y, want)), flags, pa.n_recv)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("layouts", [(0, 1), (1, 0), (0, 0)])
def test_plan_a_exchange_on_gloo_ranks(world, layouts):
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), layouts, out), nprocs=world, join=True)
    N = GRID[0] * GRID[1] * GRID[2]
    assert sum(out[r][2] for r in range(world)) == N
    for r in range(world):
        ok, flags, _ = out[r]
        assert ok, f"rank {r} ended with the wrong rows"
        assert len(set(flags)) == 1  # every rank takes the same branch
    assert out[0][1][0] == (layouts[0] != layouts[1])


def test_oracle_agrees_with_the_grid_used():
    # the oracle's simulated exchange on the same grid (cross-check of the fixture)
    src, dst = oracle.make_plan(*GRID, 0), oracle.make_plan(*GRID, 1)
    x = np.arange(src.num_tokens, dtype=np.float64)[:, None]
    got, sched = oracle.sp.simulate(x, src, dst, 3)
    for d in range(3):
        assert np.array_equal(got[d][:, 0], sched["dst_rows"][d].astype(np.float64))
