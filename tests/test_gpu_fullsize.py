"""Parity at the workloads' full sizes, in the bench's launch configuration (one
plan over the whole set).  The oracle checks sampled matrices one by one; every
matrix is checked through properties that hold at any size."""
import math

import numpy as np
import pytest

from oracle import muon_ref as R
from tests.gpu_util import LR, WD, MU, rel

pytestmark = pytest.mark.gpu

TOL_O, TOL_FP32 = 2e-2, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def device_inputs(wl, step=0):
    import torch
    import workloads
    W, G, M = [], [], []
    for i, (m, n) in enumerate(wl.shapes):
        W.append(workloads.gen_tensor((m, n), workloads.W_STD, workloads.seed_of(wl.index, 0, i, "W"), "cuda"))
        G.append(workloads.gen_tensor((m, n), workloads.G_STD, workloads.seed_of(wl.index, step, i, "G"), "cuda",
                                      wl.grad_dtype))
        M.append(workloads.gen_tensor((m, n), workloads.M_STD, workloads.seed_of(wl.index, 0, i, "M"), "cuda"))
    torch.cuda.synchronize()
    return W, G, M


def run_full(name, sample, keep_update=True):
    """One NS5 step over the whole workload; returns host copies for the sampled matrices
    plus per-matrix RMS(O) * sqrt(c) for all of them."""
    import torch
    import workloads
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    wl = workloads.WORKLOADS[name]
    W, G, M = device_inputs(wl)
    before = {i: (W[i].cpu(), G[i].cpu(), M[i].cpu()) for i in sample}
    plan = lib.MuonPlan(list(wl.shapes), wl.grad_dtype, keep_update=keep_update)
    plan.step(W, G, M, LR, WD, MU, 5, "ns")
    plan.sync()
    rms = []
    if keep_update:
        for i, (m, n) in enumerate(wl.shapes):
            o = plan.debug_update(i)
            rms.append(float(o.float().pow(2).mean().sqrt()) * math.sqrt(max(m, n)))
            assert bool(torch.isfinite(o).all()), i
    after = {i: (W[i].cpu(), M[i].cpu(), plan.debug_update(i).cpu() if keep_update else None) for i in sample}
    del W, G, M
    plan.close()
    torch.cuda.empty_cache()
    return wl, before, after, rms


def check(wl, before, after, i, o_check=True):
    w0, g, m0 = (t.double().numpy() for t in before[i])
    w1, m1, o = after[i]
    m_ref = R.momentum(m0, g, MU)
    assert rel(m1.numpy(), m_ref) <= TOL_FP32, ("M", i)
    o = o.double().numpy()
    mm, nn = wl.shapes[i]
    w_given_o = R.apply_update(w0, o, LR, WD, R.update_scale(mm, nn))
    assert rel(w1.numpy(), w_given_o) <= TOL_FP32, ("W|O", i)
    if o_check:
        o_ref = R.orthogonalised_update(R.nesterov(m_ref, g, MU), 5, form="gram")
        e = rel(o, o_ref)
        assert e <= TOL_O, ("O", i, wl.shapes[i], e)
        return e


def test_qwen7b_layer_every_matrix():
    """One Qwen2.5-7B layer: q, k, v, o, gate (T), up (T), down; every matrix vs the oracle."""
    wl, before, after, rms = run_full("qwen7b_layer", sample=list(range(7)))
    errs = [check(wl, before, after, i) for i in range(7)]
    assert all(0.6 < x < 1.2 for x in rms), rms
    print("qwen7b_layer O rel err:", ["%.2e" % e for e in errs])


def test_qwen7b_heads_every_matrix():
    """1008 matrices 128 x 3584 plus 28 transposed 3584 x 512, one plan; every matrix
    against the oracle."""
    sample = list(range(1036))
    wl, before, after, rms = run_full("qwen7b_heads", sample)
    assert len(wl.shapes) == len(sample)
    errs = [check(wl, before, after, i) for i in sample]
    assert all(0.6 < x < 1.2 for x in rms)
    print("qwen7b_heads O rel err: max %.2e" % max(errs))


def test_qwen7b_28l_layers_0_and_27():
    """The 196-matrix set of the bench: every matrix of layers 0 and 27 (O on all but the
    18944 x 3584 ones, whose shape the one-layer test checks in full), RMS band on all."""
    sample = list(range(7)) + list(range(189, 196))
    wl, before, after, rms = run_full("qwen7b_28l", sample)
    for i in sample:
        check(wl, before, after, i, o_check=wl.shapes[i] != (18944, 3584))
    assert len(rms) == 196 and all(0.6 < x < 1.2 for x in rms)


def test_dit_periodic_rownorm_8_steps():
    """28 DiT blocks, K = 4 over 8 steps with fresh grads; blocks 0 and 27 followed by the
    oracle, and at the RowNorm step t = 1 every matrix's update direction, recovered from W
    before and after, has unit oriented rows (a property of R_eps at any size)."""
    import torch
    import workloads
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    wl = workloads.WORKLOADS["dit1p3b"]
    W, G, M = device_inputs(wl)
    sample = list(range(5)) + list(range(135, 140))
    w_ref = {i: W[i].double().cpu().numpy() for i in sample}
    m_ref = {i: M[i].double().cpu().numpy() for i in sample}
    plan = lib.MuonPlan(list(wl.shapes), wl.grad_dtype)
    sched = lib.PeriodicRowNormMuon(plan, k=wl.rownorm_k, eps=wl.eps)
    for t in range(wl.steps):
        if t > 0:
            for i, (m, n) in enumerate(wl.shapes):
                G[i] = workloads.gen_tensor((m, n), workloads.G_STD, workloads.seed_of(wl.index, t, i, "G"),
                                            "cuda", wl.grad_dtype)
        w_before = [w.clone() for w in W] if t == 1 else None
        mode = sched.step(W, G, M, LR, WD)
        if w_before is not None:
            plan.sync()
            assert mode == "rownorm"
            worst = 0.0
            for i, (m, n) in enumerate(wl.shapes):
                d = ((1.0 - LR * WD) * w_before[i].double() - W[i].double()) / (LR * R.update_scale(m, n))
                norms = d.norm(dim=1) if m <= n else d.norm(dim=0)
                worst = max(worst, float((norms - 1.0).abs().max()))
            del w_before
            assert worst <= 1e-4, worst
        for i in sample:
            g = G[i].double().cpu().numpy()
            w_ref[i], m_ref[i], _ = R.muon_step(w_ref[i], g, m_ref[i], LR, WD, MU, 5, mode, wl.eps, form="gram")
    plan.sync()
    for i in sample:
        assert rel(M[i].cpu().numpy(), m_ref[i]) <= TOL_FP32, i
        mm, nn = wl.shapes[i]
        # two NS refreshes with O within 2e-2 each; RowNorm steps match to fp32
        bound = (2 * LR * R.update_scale(mm, nn) * TOL_O * math.sqrt(min(mm, nn))) / np.linalg.norm(w_ref[i])
        assert rel(W[i].cpu().numpy(), w_ref[i]) <= bound + TOL_FP32, i
