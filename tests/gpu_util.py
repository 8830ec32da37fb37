"""Helpers shared by the GPU parity tests: seeded inputs (from ``workloads``),
one library step, and oracle comparisons."""
import math

import numpy as np

from oracle import muon_ref as R
from workloads import gen_tensor, seed_of, W_STD, G_STD, M_STD

LR, WD, MU = 0.02, 0.1, 0.95


def rel(a, b):
    """||a - b||_F / ||b||_F (absolute when b is zero)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    d = np.linalg.norm(a - b)
    return float(d / nb) if nb > 0 else float(d)


def host_inputs(shapes, grad_dtype, base_seed, step=0):
    """Seeded CPU tensors (W, G, M) per matrix; G in the plan's grad dtype."""
    out = []
    for i, (m, n) in enumerate(shapes):
        w = gen_tensor((m, n), W_STD, seed_of(base_seed, 0, i, "W"))
        g = gen_tensor((m, n), G_STD, seed_of(base_seed, step, i, "G"), dtype=grad_dtype)
        mm = gen_tensor((m, n), M_STD, seed_of(base_seed, 0, i, "M"))
        out.append((w, g, mm))
    return out


def run_step(shapes, grad_dtype="bf16", base_seed=100, ns_steps=5, mode="ns", lr=LR, wd=WD, mu=MU,
             eps=1e-8, keep_update=True, inputs=None, plan=None, single_sm_gemm=False, generic_small=False,
             chain_clusters=0, workspace_bytes=0, coeffs=None, restart=0, max_ns_steps=0, small_fp32=0,
             precision=0, full_symmetric=False, precision_of=None):
    """One library step on copies of the seeded inputs; returns a dict of CPU results."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib

    if inputs is None:
        inputs = host_inputs(shapes, grad_dtype, base_seed)
    own = plan is None
    if own:
        plan = lib.MuonPlan(shapes, grad_dtype, keep_update=keep_update, single_sm_gemm=single_sm_gemm,
                            generic_small=generic_small, chain_clusters=chain_clusters,
                            workspace_bytes=workspace_bytes, max_ns_steps=max_ns_steps, small_fp32=small_fp32,
                            precision=precision, full_symmetric=full_symmetric, precision_of=precision_of)
    W = [w.cuda() for w, _, _ in inputs]
    G = [g.cuda() for _, g, _ in inputs]
    M = [m.cuda() for _, _, m in inputs]
    if mode == "ns":
        plan.step(W, G, M, lr, wd, mu, ns_steps, "ns", coeffs=coeffs, restart=restart)
    else:
        plan.rownorm_step(W, G, M, lr, wd, mu, eps)
    plan.sync()
    res = {"inputs": inputs, "W": [w.cpu() for w in W], "M": [m.cpu() for m in M], "plan": plan}
    if keep_update and mode == "ns":
        res["O"] = [plan.debug_update(i).cpu() for i in range(len(shapes))]
    return res


def oracle_step(inp, lr=LR, wd=WD, mu=MU, ns_steps=5, mode="ns", eps=1e-8):
    w, g, m = (t.double().numpy() for t in inp)
    return R.muon_step(w, g, m, lr, wd, mu, ns_steps, mode, eps)


def check_ns_matrix(res, i, ns_steps=5, tol_o=2e-2, lr=LR, wd=WD, mu=MU):
    """The bars of the method on one matrix: M and W-given-O to 1e-5, O to tol_o."""
    inp = res["inputs"][i]
    w_ref, m_ref, o_ref = oracle_step(inp, lr, wd, mu, ns_steps)
    e_m = rel(res["M"][i].numpy(), m_ref)
    o_gpu = res["O"][i].double().numpy()
    e_o = rel(o_gpu, o_ref)
    m_, n_ = o_gpu.shape
    w_given_o = R.apply_update(inp[0].double().numpy(), o_gpu, lr, wd, R.update_scale(m_, n_))
    e_w = rel(res["W"][i].numpy(), w_given_o)
    # end to end: an O error of tol_o moves W by at most lr * s * tol_o * ||O||
    bound = (lr * R.update_scale(m_, n_) * tol_o * np.linalg.norm(o_ref)
             + 1e-6 * np.linalg.norm(w_ref)) / np.linalg.norm(w_ref)
    e_we = rel(res["W"][i].numpy(), w_ref)
    return dict(m=e_m, o=e_o, w_given_o=e_w, w_e2e=e_we, w_bound=bound)


def check_rownorm_matrix(res, i, lr=LR, wd=WD, mu=MU, eps=1e-8):
    inp = res["inputs"][i]
    w_ref, m_ref, _ = oracle_step(inp, lr, wd, mu, 0, "rownorm", eps)
    return dict(m=rel(res["M"][i].numpy(), m_ref), w=rel(res["W"][i].numpy(), w_ref))


def nesterov_u(inp, mu=MU):
    _, g, m = (t.double().numpy() for t in inp)
    m1 = R.momentum(m, g, mu)
    return R.nesterov(m1, g, mu)


def fro(x):
    return math.sqrt(float(np.sum(np.asarray(x, np.float64) ** 2)))
