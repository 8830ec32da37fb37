"""Owner partition across ranks on CPU: the library's muon_partition (host only)
and DistributedMuon's exchange over two gloo ranks.  The ranks' local step here
is the fp64 oracle (test infrastructure, injected by subclassing), so what is
tested is the partition and the parameter exchange: every rank ends with the
same parameters as one process stepping every matrix."""
import os
import socket

import numpy as np
import pytest

import matrix_orthogonalising_optimizer_muon_gb300 as mu


def test_partition_is_lpt_on_given_costs():
    """Longest processing time first, ties by index and by rank: on costs 5, 4, 3, 3, 3
    over two ranks it gives loads 8 and 10 (the optimum, 9 and 9, is not what LPT finds)."""
    shapes = [(8, 8)] * 5
    owners, loads = mu.partition_owners(shapes, 2, costs=[5, 4, 3, 3, 3])
    assert owners == [0, 1, 1, 0, 1]
    assert loads == [8.0, 10.0]
    owners, loads = mu.partition_owners(shapes, 1, costs=[5, 4, 3, 3, 3])
    assert owners == [0] * 5 and loads == [18.0]
    # more ranks than matrices: one matrix each, the rest idle
    owners, loads = mu.partition_owners(shapes[:3], 5, costs=[1, 2, 3])
    assert owners == [2, 1, 0] and loads == [3.0, 2.0, 1.0, 0.0, 0.0]


@pytest.mark.parametrize("world", [2, 3, 8])
def test_partition_of_the_28_layer_set_covers_and_balances(world):
    import workloads
    shapes = list(workloads.WORKLOADS["qwen7b_28l"].shapes)
    owners, loads = mu.partition_owners(shapes, world)
    assert len(owners) == len(shapes) and all(0 <= o < world for o in owners)
    assert mu.partition_owners(shapes, world) == (owners, loads)   # deterministic
    per = [sum(1 for o in owners if o == r) for r in range(world)]
    assert sum(per) == len(shapes) and min(per) > 0
    # the model's costs: the loads sum to the total and LPT keeps max - min below the largest cost
    costs = []
    for m, n in shapes:
        r, c = min(m, n), max(m, n)
        costs.append(max(24.0 * r * c / 6.8e12, (3.0 * r * r * c + 17.0 * r ** 3) / 1.5e15))
    assert abs(sum(loads) - sum(costs)) < 1e-9 * sum(costs)
    assert max(loads) - min(loads) <= max(costs) * (1 + 1e-9)
    for r in range(world):
        assert abs(loads[r] - sum(c for c, o in zip(costs, owners) if o == r)) < 1e-12


def test_partition_rejects_bad_arguments():
    with pytest.raises(mu.MuonError):
        mu.partition_owners([(8, 8)], 0)
    with pytest.raises(mu.MuonError):
        mu.partition_owners([(8, 8), (4, 4)], 2, costs=[1.0, -1.0])
    with pytest.raises(mu.MuonError):
        mu.partition_owners([(8, 8)], 2, costs=[float("nan")])
    with pytest.raises(mu.MuonError):
        mu.partition_owners([(0, 8)], 2)


# ---------------------------------------------------------------- two gloo ranks
SHAPES = [(32, 48), (48, 32), (16, 64), (64, 16), (24, 24), (40, 56), (8, 8)]
LR, WD, MU = 0.02, 0.1, 0.95


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs(step):
    from workloads import gen_tensor, seed_of
    W = [gen_tensor(s, 0.02, seed_of(70, 0, i, "W")) for i, s in enumerate(SHAPES)]
    M = [gen_tensor(s, 1e-3, seed_of(70, 0, i, "M")) for i, s in enumerate(SHAPES)]
    G = [[gen_tensor(s, 1e-3, seed_of(70, t, i, "G")) for i, s in enumerate(SHAPES)] for t in range(step)]
    return W, M, G


class OracleOwners(mu.DistributedMuon):
    """The owner partition and exchange of DistributedMuon with the fp64 oracle as each
    rank's local step (CPU tensors, no CUDA library)."""

    def _make_plan(self, plan_opts):
        return None

    def _local_step(self, params, grads, momentum, lr, wd, mu_, ns_steps, mode, eps, stream):
        from oracle import muon_ref as R
        for w, g, m in zip(params, grads, momentum):
            w2, m2, _ = R.muon_step(w.double().numpy(), g.double().numpy(), m.double().numpy(), lr, wd, mu_,
                                    ns_steps, mode, eps)
            w.copy_(__import__("torch").from_numpy(w2))
            m.copy_(__import__("torch").from_numpy(m2))


MODES = ["ns", "rownorm", "ns"]


def _worker(rank, world, port, in_place, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    opt = OracleOwners(SHAPES, "f32")
    W0, M0, G = _inputs(len(MODES))
    if in_place:
        W = opt.allocate_params("cpu")
        for w, w0 in zip(W, W0):
            w.copy_(w0)
    else:
        W = [w.clone() for w in W0]
    # momentum only where this rank owns the matrix
    M = [M0[i].clone() if i in opt.owned else None for i in range(len(SHAPES))]
    for t, mode in enumerate(MODES):
        grads = [G[t][i] if i in opt.owned else None for i in range(len(SHAPES))]
        opt.step(W, grads, M, LR, WD, MU, 5, mode)
    out[rank] = {"owner": list(opt.owner), "W": [w.numpy().copy() for w in W],
                 "M": {i: M[i].numpy().copy() for i in opt.owned}}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("in_place", [True, False], ids=["flat_params", "staged"])
def test_two_gloo_ranks_match_one_process_bitwise(in_place):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _free_port(), in_place, out), nprocs=2, join=True, start_method="spawn")
    res = dict(out)
    owners = res[0]["owner"]
    assert owners == res[1]["owner"] and set(owners) == {0, 1}
    # one process stepping every matrix with the same local step
    from oracle import muon_ref as R
    W0, M0, G = _inputs(len(MODES))
    W = [w.double().numpy() for w in W0]
    M = [m.double().numpy() for m in M0]
    for t, mode in enumerate(MODES):
        for i in range(len(SHAPES)):
            w2, m2, _ = R.muon_step(W[i], G[t][i].double().numpy(), M[i], LR, WD, MU, 5, mode)
            W[i] = np.float32(w2).astype(np.float64)
            M[i] = np.float32(m2).astype(np.float64)
    for rank in (0, 1):
        for i in range(len(SHAPES)):
            assert np.array_equal(res[rank]["W"][i], np.float32(W[i])), (rank, i)
        for i, m in res[rank]["M"].items():
            assert owners[i] == rank and np.array_equal(m, np.float32(M[i])), (rank, i)
    assert set(res[0]["M"]) | set(res[1]["M"]) == set(range(len(SHAPES)))


# ---------------------------------------------------------------- sharded RowNorm over two gloo ranks
FULL = [(64, 24), (24, 64), (48, 48), (130, 20), (20, 130)]   # full shapes (m, n)


class OracleShards(mu.ShardedRowNorm):
    """ShardedRowNorm's step (statistics, all-reduce, update) with fp64 CPU arithmetic as
    each rank's local part, written from the RowNorm definition: R(U)_i = U_i / max(||U_i||,
    eps) over the rows of the oriented full matrix (stored columns when m > n)."""

    def _make_plan(self, shard_shapes, full_rows, grad_dtype, plan_opts):
        self.shapes, self.full_rows = shard_shapes, full_rows
        return None

    def _colsq_len(self):
        return sum((n + 3) // 4 * 4 for (m, n), f in zip(self.shapes, self.full_rows) if f > n)

    def _device(self):
        return "cpu"

    def _stats(self, params, grads, momentum, lr, wd, mu_, eps, stream):
        import torch
        self.colsq = self.colsq.double()
        off = 0
        for (m, n), f, w, g, mo in zip(self.shapes, self.full_rows, params, grads, momentum):
            mo.mul_(mu_).add_(g)                   # M <- mu M + G
            u = mu_ * mo + g
            scale = 0.2 * (max(f, n) ** 0.5)
            if f <= n:                             # every RowNorm row is complete here
                r = u / torch.clamp(u.norm(dim=1, keepdim=True), min=eps)
                w.sub_(lr * (scale * r + wd * w))
            else:
                self.colsq[off:off + n] = (u * u).sum(dim=0)
                off += (n + 3) // 4 * 4

    def _apply(self, params, grads, momentum, lr, wd, mu_, eps, stream):
        import torch
        off = 0
        for (m, n), f, w, g, mo in zip(self.shapes, self.full_rows, params, grads, momentum):
            if f <= n:
                continue
            u = mu_ * mo + g
            inv = 1.0 / torch.clamp(self.colsq[off:off + n].sqrt(), min=eps)
            w.sub_(lr * (0.2 * (max(f, n) ** 0.5) * u * inv + wd * w))
            off += (n + 3) // 4 * 4


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    from workloads import gen_tensor, seed_of
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shard_shapes, params, grads, moms = [], [], [], []
    for i, (m, n) in enumerate(FULL):
        lo, hi = rank * m // world, (rank + 1) * m // world   # dim-0 shard of the full matrix
        w = gen_tensor((m, n), 0.02, seed_of(72, 0, i, "W")).double()
        g = gen_tensor((m, n), 1e-3, seed_of(72, 0, i, "G")).double()
        mm = gen_tensor((m, n), 1e-3, seed_of(72, 0, i, "M")).double()
        shard_shapes.append((hi - lo, n))
        params.append(w[lo:hi].clone())
        grads.append(g[lo:hi].clone())
        moms.append(mm[lo:hi].clone())
    opt = OracleShards(shard_shapes, [m for m, _ in FULL], "f32")
    opt.step(params, grads, moms, LR, WD, MU, 1e-8)
    out[rank] = [p.numpy().copy() for p in params]
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_rownorm_over_two_gloo_ranks_matches_the_full_oracle():
    """Two ranks each hold half of the rows of every matrix; one sharded RowNorm step
    (local statistics, one all-reduce of the column sums, local update) gives the oracle's
    RowNorm step on the full matrices."""
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    from oracle import muon_ref as R
    from workloads import gen_tensor, seed_of
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_shard_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    for i, (m, n) in enumerate(FULL):
        w = gen_tensor((m, n), 0.02, seed_of(72, 0, i, "W")).double().numpy()
        g = gen_tensor((m, n), 1e-3, seed_of(72, 0, i, "G")).double().numpy()
        mm = gen_tensor((m, n), 1e-3, seed_of(72, 0, i, "M")).double().numpy()
        w_ref, _, _ = R.muon_step(w, g, mm, LR, WD, MU, 0, "rownorm", 1e-8)
        got = np.concatenate([out[0][i], out[1][i]], axis=0)
        assert np.abs(got - w_ref).max() <= 1e-12 * np.abs(w_ref).max(), (i, (m, n))
