"""The N > 1 bench path on CPU: two gloo ranks (replicas), barrier and the
max-over-ranks timing reduction used for the reported step time."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's "step time" differs; every rank must see the max
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_over_ranks():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("gloo path is exercised on CPU-only hosts")
    import torch.multiprocessing as mp
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_flop_accounting_matches_gram_form():
    import bench
    # one 3584 x 18944 matrix, J = 5: 3 r^2 c (r x c products) + 17 r^3 (r x r products)
    rc, rrr = bench.algorithmic_ns_flops([(18944, 3584)], 5)
    r, c = 3584, 18944
    assert rc == 3.0 * r * r * c and rrr == 17.0 * r ** 3
    assert bench.algorithmic_ns_flops([(8, 16)], 1) == (3.0 * 64 * 16, 512.0)
    assert bench.algorithmic_ns_flops([(8, 16)], 0)[1] == 0.0
