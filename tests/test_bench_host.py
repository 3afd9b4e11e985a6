"""CPU tests of bench.py's host logic: algorithmic byte/FLOP counts and the
multi-rank (replica) aggregation over a world-size-2 gloo group."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from gated_deltanet_linear_fwd_gb300.inputs import make_inputs


def test_algorithmic_counts_match_hand_figures():
    # 1 x 32768, h_qk = 2, h_v = 8: q,k 33.6 MB, v,o 134.2 MB, g,beta 2.1 MB, final state 0.5 MB
    w = make_inputs(32768, h_qk=2, h_v=8, seed=1)
    by, fl = bench.algorithmic(w)
    assert by == 32768 * (2 * 2 * 128 * 2 + 2 * 8 * 128 * 2 + 2 * 8 * 4) + 8 * 128 * 128 * 4
    assert abs(by / 1e6 - 170.4) < 0.1
    assert abs(fl / 1e9 - 41.16) < 0.05


def test_kernel_bytes_partition_the_layer_bytes():
    # the WY kernel's reads plus the output scan's writes are exactly the layer's algorithmic bytes
    for kw in (dict(with_h0=False), dict(with_h0=True)):
        w = make_inputs(4096, h_qk=2, h_v=8, seed=1, **kw)
        by, _ = bench.algorithmic(w)
        assert bench.kernel_bytes("wy", w) + bench.kernel_bytes("scan_out", w) == by
        assert bench.kernel_bytes("combine", w) == bench.kernel_bytes("scan_prep", w) == 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w, "cpu")
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo replica path is checked on CPU-only hosts")
def test_replica_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5
