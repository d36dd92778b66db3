"""The column split over N (the GLU segment under column-parallel gate/up
projections): every rank streams its rows of both weights and writes its
columns of out, with no collective on the data path.  CPU only: the shares
cover [0, N) exactly, and shard-wise oracle results, gathered here by the
test over gloo (world size 2), concatenate bit for bit to the whole-N result
-- for glu_gemv, and for add_rmsnorm_glu, whose prologue every rank repeats
(its residual update is then identical on every rank)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import glu_inputs as gi
import oracle
from memory_bound_glu_gb300.binding import column_shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("N", [0, 1, 5, 8, 3072, 9728, 11008, 14336])
def test_shares_partition_the_rows(N, world):
    shares = [column_shard(N, world, p) for p in range(world)]
    assert shares[0][0] == 0 and shares[-1][1] == N
    for (a, b), (c, d) in zip(shares, shares[1:]):
        assert b == c and a <= b
    sizes = [b - a for a, b in shares]
    assert max(sizes) - min(sizes) <= 1


def test_bad_split_is_rejected():
    for args in ((10, 0, 0), (10, 2, 2), (10, 2, -1), (-1, 2, 0)):
        with pytest.raises(ValueError):
            column_shard(*args)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


M, N, K = 3, 1001, 512


def _operands():
    h = gi.bits(gi.normal_bf16((M, K), 1.0, 4, "cs-h"))
    g = gi.bits(gi.normal_bf16((N, K), K ** -0.5, 4, "cs-g"))
    u = gi.bits(gi.normal_bf16((N, K), K ** -0.5, 4, "cs-u"))
    x = gi.bits(gi.normal_bf16((M, K), 1.0, 4, "cs-x"))
    r = gi.bits(gi.normal_bf16((M, K), 1.0, 4, "cs-r"))
    w = gi.bits(gi.normal_bf16((K,), 0.1, 4, "cs-w"))
    return h, g, u, x, r, w


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    h, g, u, x, r, w = _operands()
    lo, hi = column_shard(N, world, rank)
    out = oracle.glu_gemv(h, np.ascontiguousarray(g[lo:hi]), np.ascontiguousarray(u[lo:hi]), "hf", nthreads=1)
    nout, res, _ = oracle.add_rmsnorm_glu(x, r, w, 1e-6, np.ascontiguousarray(g[lo:hi]),
                                          np.ascontiguousarray(u[lo:hi]), "hf", nthreads=1)
    # the test gathers the shards to check them; the split itself needs no collective
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, out, nout, res))
    if rank == 0:
        q.put(parts)
    dist.destroy_process_group()


def test_shards_concatenate_to_the_whole_result_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(p, world, port, q)) for p in range(world)]
    for p in procs:
        p.start()
    parts = q.get(timeout=180)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    h, g, u, x, r, w = _operands()
    whole = oracle.glu_gemv(h, g, u, "hf", nthreads=1)
    nwhole, res_whole, _ = oracle.add_rmsnorm_glu(x, r, w, 1e-6, g, u, "hf", nthreads=1)
    assert [(a, b) for a, b, *_ in parts] == [column_shard(N, world, p) for p in range(world)]
    assert np.array_equal(np.concatenate([p[2] for p in parts], axis=1), whole)
    assert np.array_equal(np.concatenate([p[3] for p in parts], axis=1), nwhole)
    for p in parts:   # every rank repeats the prologue: the same residual update
        assert np.array_equal(p[4], res_whole)
