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
    """28 DiT blocks, K = 4 over 8 steps with fresh grads; blocks 0, 13 and 27 followed by the
    oracle, and at the RowNorm step t = 1 every matrix's update direction, recovered from W
    before and after, has unit oriented rows (a property of R_eps at any size)."""
    import torch
    import workloads
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    wl = workloads.WORKLOADS["dit1p3b"]
    W, G, M = device_inputs(wl)
    sample = list(range(5)) + list(range(65, 70)) + list(range(135, 140))
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


def test_qwen7b_28l_one_matrix_per_shape_per_layer():
    """The 196-matrix set: in every layer one randomly chosen matrix of each oriented
    shape (q / o 3584 x 3584, k / v 512 x 3584, gate / up / down 3584 x 18944): momentum
    and W given O at 1e-5 (the 3584 x 18944 ones in seven random layers, the others in
    all 28), O against the oracle for the 512 x 3584 ones of every layer and the
    3584 x 3584 ones of three random layers.  Inputs are regenerated from their seeds
    after the step, so no host copy of the whole set is kept."""
    import torch
    import workloads
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    wl = workloads.WORKLOADS["qwen7b_28l"]
    rng = np.random.default_rng(2028)
    within = {"sq": (0, 3), "kv": (1, 2), "ffn": (4, 5, 6)}   # q, k, v, o, gate, up, down
    ffn_layers = set(rng.choice(28, 7, replace=False).tolist())
    o_sq_layers = set(rng.choice(28, 3, replace=False).tolist())
    picks = [(layer, kind, 7 * layer + int(rng.choice(idx))) for layer in range(28) for kind, idx in within.items()]
    W, G, M = device_inputs(wl)
    plan = lib.MuonPlan(list(wl.shapes), wl.grad_dtype, keep_update=True)
    plan.step(W, G, M, LR, WD, MU, 5, "ns")
    plan.sync()
    worst = {"m": 0.0, "w": 0.0, "o": 0.0}
    for layer, kind, i in picks:
        if kind == "ffn" and layer not in ffn_layers:
            continue
        shape = wl.shapes[i]

        def seeded(kind_, std, dtype="f32"):
            t = workloads.gen_tensor(shape, std, workloads.seed_of(wl.index, 0, i, kind_), "cuda", dtype)
            return t.double().cpu().numpy()

        w0, g, m0 = seeded("W", workloads.W_STD), seeded("G", workloads.G_STD, wl.grad_dtype), seeded("M", workloads.M_STD)
        m_ref = R.momentum(m0, g, MU)
        e_m = rel(M[i].cpu().numpy(), m_ref)
        o = plan.debug_update(i).cpu().double().numpy()
        e_w = rel(W[i].cpu().numpy(), R.apply_update(w0, o, LR, WD, R.update_scale(*shape)))
        assert e_m <= TOL_FP32 and e_w <= TOL_FP32, (layer, kind, i, e_m, e_w)
        worst["m"], worst["w"] = max(worst["m"], e_m), max(worst["w"], e_w)
        if kind == "kv" or (kind == "sq" and layer in o_sq_layers):
            e_o = rel(o, R.orthogonalised_update(R.nesterov(m_ref, g, MU), 5, form="gram"))
            assert e_o <= TOL_O, (layer, kind, i, e_o)
            worst["o"] = max(worst["o"], e_o)
    del W, G, M
    plan.close()
    torch.cuda.empty_cache()
    print("qwen7b_28l sampled per layer:", {k: "%.2e" % v for k, v in worst.items()})
