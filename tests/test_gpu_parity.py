"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on seeded
inputs.  Bars: relative Frobenius error <= 2e-2 on the orthogonalised update O
(bf16/fp16 tensor-core path) and <= 1e-5 on momentum, on weights given the
GPU's own O, and on RowNorm outputs."""
import numpy as np
import pytest

from oracle import muon_ref as R
from tests.gpu_util import (LR, WD, MU, check_ns_matrix, check_rownorm_matrix, host_inputs,
                            nesterov_u, rel, run_step)

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_FP32 = 1e-5


def lib_scale(r):
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    return lib.MuonPlan.gram_scale(r)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    lib.load()


def assert_ns(res, i, tol_o=TOL_O, ns_steps=5):
    e = check_ns_matrix(res, i, ns_steps, tol_o)
    assert e["m"] <= TOL_FP32, (i, e)
    assert e["o"] <= tol_o, (i, e)
    assert e["w_given_o"] <= TOL_FP32, (i, e)
    assert e["w_e2e"] <= e["w_bound"], (i, e)
    return e


# --------------------------------------------------------------- stage by stage
def test_stages_ns0_x0_alpha_gram_and_final_product():
    """ns_steps = 0: X0 workspace (momentum kernels), 1/||U||, G0 (SYRK, bf16 K-major
    operands) and O = X0 through the final product (MN-major bf16 operand)."""
    shapes = [(300, 700), (700, 300), (128, 256)]
    res = run_step(shapes, "bf16", base_seed=11, ns_steps=0, generic_small=True)
    plan = res["plan"]
    for i, (m, n) in enumerate(shapes):
        u = nesterov_u(res["inputs"][i])
        ut, _ = R.orient(u)
        x_ws = plan.debug_workspace(i, 0).double().numpy()
        # bf16 round-to-nearest of the fp32 U: within one bf16 half-ulp (+fp32 noise)
        assert np.all(np.abs(x_ws - ut) <= np.abs(ut) * (2.0 ** -8) + 1e-30), i
        alpha = float(plan.debug_workspace(i, 8)[0])
        assert abs(alpha * np.linalg.norm(u) - 1) < 1e-5, i
        sc = lib_scale(min(m, n))
        g0 = plan.debug_workspace(i, 1).double().numpy() / sc
        g_ref = (x_ws @ x_ws.T) * alpha ** 2           # from the GPU's own bf16 operand
        assert rel(g0, g_ref) < 2e-3, i
        assert np.array_equal(g0, g0.T), i             # mirrored lower triangle
        qb = plan.debug_workspace(i, 7).double().numpy()
        assert np.array_equal(qb, np.eye(min(m, n))), i
        e = assert_ns(res, i, tol_o=1e-2, ns_steps=0)
        assert e["o"] < 1e-2


def test_stages_ns1_polynomial_epilogue():
    """ns_steps = 1: P1 = aI + bG0 + cG0^2 (fp16 product + polynomial epilogue)."""
    shapes = [(384, 1000), (1000, 384)]
    res = run_step(shapes, "bf16", base_seed=12, ns_steps=1, generic_small=True)
    plan = res["plan"]
    a, b, c = R.NS_COEFFS
    for i in range(len(shapes)):
        g0 = plan.debug_workspace(i, 1).double().numpy() / lib_scale(min(shapes[i]))
        p1 = plan.debug_workspace(i, 3).double().numpy()
        r = g0.shape[0]
        p_ref = a * np.eye(r) + b * g0 + c * (g0 @ g0)
        assert rel(p1, p_ref) < 2e-3, i
        qb = plan.debug_workspace(i, 7).double().numpy()
        assert rel(qb, p_ref) < 1e-2, i
        assert_ns(res, i, ns_steps=1)


def test_stages_ns2_products():
    """ns_steps = 2: T = P1 P1, G1 = G0 T, Q2 = P2 P1 (all fp16 symmetric products)."""
    shapes = [(256, 640)]
    res = run_step(shapes, "f32", base_seed=13, ns_steps=2, generic_small=True)
    plan = res["plan"]
    a, b, c = R.NS_COEFFS
    sc = lib_scale(256)
    g0 = plan.debug_workspace(0, 1).double().numpy() / sc
    r = g0.shape[0]
    p1 = a * np.eye(r) + b * g0 + c * g0 @ g0
    t = plan.debug_workspace(0, 4).double().numpy()
    assert rel(t, p1 @ p1) < 3e-3
    g1 = plan.debug_workspace(0, 2).double().numpy() / sc
    assert rel(g1, g0 @ p1 @ p1) < 5e-3
    p2 = plan.debug_workspace(0, 3).double().numpy()
    assert rel(p2, a * np.eye(r) + b * g1 + c * g1 @ g1) < 3e-3
    qb = plan.debug_workspace(0, 7).double().numpy()
    assert rel(qb, p2 @ p1) < 1e-2
    assert_ns(res, 0, ns_steps=2)


# --------------------------------------------------------------- full steps
def test_single_256x1024_fp32_grads():
    """The 256 x 1024 single-matrix workload (fp32 W, G, M; seed 0)."""
    import workloads
    wl = workloads.WORKLOADS["single"]
    inputs = [workloads.matrix_inputs(wl, 0, 0)]
    res = run_step(list(wl.shapes), "f32", inputs=inputs)
    e = assert_ns(res, 0)
    assert e["o"] < 1e-2


RAGGED = [(7, 13), (13, 7), (130, 300), (300, 130), (384, 384), (129, 1000), (1000, 129),
          (1, 64), (64, 1), (256, 1024), (520, 2100)]


@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_mixed_ragged_plan_ns5(grad_dtype):
    """Many buckets in one plan, ragged tails in every dimension, both orientations."""
    res = run_step(RAGGED, grad_dtype, base_seed=21)
    for i in range(len(RAGGED)):
        assert_ns(res, i)


def test_single_sm_kernel_ns5():
    """The same mixed plan on the one-SM kernel only (128 x 256 tiles, cta_group::1):
    both tensor-core kernels stay at the oracle's bar, and agree with each other."""
    pair = run_step(RAGGED, "bf16", base_seed=26)
    single = run_step(RAGGED, "bf16", base_seed=26, single_sm_gemm=True)
    for i in range(len(RAGGED)):
        assert_ns(single, i)
        assert rel(single["O"][i].numpy(), pair["O"][i].double().numpy()) < 2e-3, RAGGED[i]


# Rectangular shapes (c >= 1.25 r) on the fused tensor-core kernel.  Nearly square ones
# (c < 1.25 r) take the fp32 kernel by default (test_small_square_fp32_path below).
SMALL = [(128, 3584), (3584, 128), (7, 13), (13, 7), (1, 64), (64, 1), (100, 1000), (128, 160), (65, 300),
         (300, 65), (128, 200)]


@pytest.mark.parametrize("ns_steps", [0, 1, 2, 5])
def test_fused_small_kernel(ns_steps):
    """r <= 128: the whole step of each matrix runs in the fused one-SM kernel (SYRK,
    on-chip recursion, final product + update); checked against the oracle and
    against the batched products of the same plan."""
    fused = run_step(SMALL, "bf16", base_seed=28, ns_steps=ns_steps)
    generic = run_step(SMALL, "bf16", base_seed=28, ns_steps=ns_steps, generic_small=True)
    for i in range(len(SMALL)):
        assert_ns(fused, i, ns_steps=ns_steps)
        assert rel(fused["O"][i].numpy(), generic["O"][i].double().numpy()) < TOL_O, SMALL[i]


SQUARE = [(16, 16), (64, 64), (96, 96), (100, 100), (128, 128), (64, 72), (140, 128), (7, 8)]


@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_small_square_fp32_path(grad_dtype):
    """Nearly square matrices with r <= 128 run the whole step in fp32 (default
    small_fp32 = 0), inside a plan that also holds fused, batched and larger square
    matrices: O within the 2e-2 bar, and in fact within 1e-3 (fp32 arithmetic)."""
    shapes = SQUARE + [(128, 3584), (300, 700), (384, 384)]
    res = run_step(shapes, grad_dtype, base_seed=30)
    for i in range(len(SQUARE)):
        e = assert_ns(res, i)
        assert e["o"] <= 1e-3, (shapes[i], e)
    for i in range(len(SQUARE), len(shapes)):
        assert_ns(res, i)


@pytest.mark.parametrize("ns_steps", [0, 1, 2, 5])
def test_fp32_path_step_counts_and_generic_small(ns_steps):
    """The fp32 kernel at J = 0, 1, 2, 5; generic_small does not move these matrices to
    the fp16 products (so both settings meet the bar)."""
    for generic in (False, True):
        res = run_step(SQUARE, "bf16", base_seed=31, ns_steps=ns_steps, generic_small=generic)
        for i in range(len(SQUARE)):
            e = assert_ns(res, i, ns_steps=ns_steps)
            assert e["o"] <= 1e-3, (SQUARE[i], generic, e)


def test_fp32_path_for_every_small_matrix_and_coefficients():
    """small_fp32 = 1: rectangular r <= 128 matrices also run in fp32 (here long ones and
    both orientations), with the pages' and the cubic coefficients."""
    shapes = [(128, 3584), (3584, 128), (100, 1000), (13, 7), (96, 96)]
    for coeffs in (None, (1.5, -0.5, 0.0)):
        res = run_step(shapes, "bf16", base_seed=32, small_fp32=1, coeffs=coeffs)
        for i in range(len(shapes)):
            e = check_ns_variant(res, i, 5, coeffs or R.NS_COEFFS, 1e-3)
            assert e <= 1e-3, (shapes[i], coeffs, e)


def test_small_square_tensor_core_paths_documented_bound():
    """small_fp32 = -1 keeps nearly square r <= 128 matrices on the tensor cores (fused
    kernel, or the batched products with generic_small): bf16 X0 and Q with the fp16 Gram
    recursion put their O at 1.3e-2 to 8e-2 (emulated; the quintic amplifies the
    near-zero singular directions by about 485), so the bound pinned here is 1e-1;
    momentum and W-given-O keep 1e-5."""
    shapes = [(96, 96), (128, 128), (64, 64)]
    for generic in (False, True):
        res = run_step(shapes, "bf16", base_seed=30, generic_small=generic, small_fp32=-1)
        for i in range(len(shapes)):
            e = check_ns_matrix(res, i, 5, 1e-1)
            assert e["o"] <= 1e-1 and e["m"] <= TOL_FP32 and e["w_given_o"] <= TOL_FP32, (shapes[i], generic, e)


def test_fused_small_kernel_batched():
    """Many r = 128 matrices (the per-head shape) across a persistent grid, plus one
    larger bucket in the same plan."""
    shapes = [(128, 3584)] * 200 + [(3584, 512)] * 2
    res = run_step(shapes, "bf16", base_seed=29)
    for i in [0, 1, 57, 199, 200, 201]:
        assert_ns(res, i)


@pytest.mark.parametrize("ns_steps", [1, 2])
def test_fused_small_w_staging_waits_for_last_epilogue(ns_steps):
    """Many short fused matrices per CTA at one and two NS steps, three steps on one plan;
    every matrix's W must equal W0 updated with its own O.  With one step the last on-chip
    epilogue reads G' and writes P in the shared-memory buffers that the W staging of the
    final phase reuses; the epilogue warps meet on an mbarrier before staging.  Without it
    W went wrong only when the W pieces came from L2 within a few hundred cycles (a kernel
    that prefetched W into L2 during the recursion); on plain inputs the window is too short
    to open, so this is a regression guard, not a reproducer."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(128, 256)] * 120 + [(100, 200)] * 100 + [(64, 128)] * 100
    plan = lib.MuonPlan(shapes, "bf16", keep_update=True)
    try:
        for seed in (33, 34, 35):
            res = run_step(shapes, "bf16", base_seed=seed, ns_steps=ns_steps, plan=plan)
            for i in range(len(shapes)):
                o = res["O"][i].double().numpy()
                m_, n_ = o.shape
                w0 = res["inputs"][i][0].double().numpy()
                w_given_o = R.apply_update(w0, o, LR, WD, R.update_scale(m_, n_))
                assert rel(res["W"][i].numpy(), w_given_o) <= TOL_FP32, (seed, i, shapes[i])
        for i in [0, 119, 120, 219, 220, 319]:
            assert_ns(res, i, ns_steps=ns_steps)
    finally:
        plan.close()


def test_batched_bucket_ns5():
    """Several same-shape matrices batched in one bucket (grouped launch items)."""
    shapes = [(200, 520)] * 5 + [(520, 200)] * 3
    res = run_step(shapes, "bf16", base_seed=22)
    for i in range(len(shapes)):
        assert_ns(res, i)


@pytest.mark.parametrize("ns_steps", [3, 4])
def test_other_ns_step_counts(ns_steps):
    res = run_step([(192, 576), (576, 192)], "bf16", base_seed=23, ns_steps=ns_steps)
    for i in range(2):
        assert_ns(res, i, ns_steps=ns_steps)


# Measured O errors of the rank-3 inputs below on GB300 (precision 0), by (J, generic_small):
# (3, fused) 0.068-0.083, (3, batched) 0.081-0.089, (5, fused) 0.90-1.85, (5, batched) 1.85-2.61.
RANK3_BOUND = {3: 0.12, 5: 3.4}


@pytest.mark.parametrize("ns_steps", [3, 5])
@pytest.mark.parametrize("generic_small", [False, True])
def test_rank_deficient_input_stays_finite(ns_steps, generic_small):
    """U of rank 3 < r.  NS amplifies small singular values by design (about a^J near
    0), and bf16 rounding of X0 leaves ~1e-4 singular values in U's null space, so a
    bf16 NS of an exactly low-rank U is not close to the exact one (the fp64 oracle
    maps those directions to 0).  What must hold up to the largest supported J (5):
    no NaN or inf, O bounded, O within the measured error plus 30 %, and the momentum
    and the update given O exact."""
    import torch
    shapes = [(96, 300), (300, 96), (200, 700)]
    inputs = []
    for i, (m, n) in enumerate(shapes):
        w, _, mo = host_inputs([(m, n)], "f32", 27 + i)[0]
        gen = torch.Generator().manual_seed(27 + i)
        low = torch.randn(m, 3, generator=gen) @ torch.randn(3, n, generator=gen) * 1e-3
        inputs.append((w, low, torch.zeros_like(mo)))
    res = run_step(shapes, "f32", inputs=inputs, ns_steps=ns_steps, generic_small=generic_small)
    for i in range(len(shapes)):
        assert bool(torch.isfinite(res["O"][i]).all()) and bool(torch.isfinite(res["W"][i]).all()), shapes[i]
        assert float(res["O"][i].abs().max()) < 1.0, shapes[i]
        e = check_ns_matrix(res, i, ns_steps, RANK3_BOUND[ns_steps])
        assert e["o"] <= RANK3_BOUND[ns_steps], (shapes[i], e)
        assert e["m"] <= TOL_FP32 and e["w_given_o"] <= TOL_FP32, (shapes[i], e)


def test_zero_input_gives_weight_decay_only():
    import torch
    shapes = [(64, 160), (160, 64)]
    inputs = [(w, torch.zeros_like(g), torch.zeros_like(m)) for w, g, m in host_inputs(shapes, "bf16", 24)]
    res = run_step(shapes, "bf16", inputs=inputs)
    for i in range(2):
        assert float(res["O"][i].abs().max()) == 0.0
        w0 = inputs[i][0].double().numpy()
        assert rel(res["W"][i].numpy(), (1 - LR * WD) * w0) < 1e-6


def test_deterministic():
    shapes = [(300, 700), (700, 300)]
    a = run_step(shapes, "bf16", base_seed=25, keep_update=False)
    b = run_step(shapes, "bf16", base_seed=25, keep_update=False)
    for i in range(2):
        assert np.array_equal(a["W"][i].numpy(), b["W"][i].numpy())
        assert np.array_equal(a["M"][i].numpy(), b["M"][i].numpy())


# --------------------------------------------------------------- RowNorm
ROWNORM_SHAPES = [(7, 13), (13, 7), (256, 1024), (1024, 256), (130, 20000), (20000, 130), (96, 96),
                  (33, 4097)]


@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_rownorm_step(grad_dtype):
    res = run_step(ROWNORM_SHAPES, grad_dtype, base_seed=31, mode="rownorm", keep_update=False)
    for i in range(len(ROWNORM_SHAPES)):
        e = check_rownorm_matrix(res, i)
        assert e["m"] <= TOL_FP32 and e["w"] <= TOL_FP32, (ROWNORM_SHAPES[i], e)


# m > n matrices of the column path (statistics, finalize, apply): column counts past a
# multiple of the blocks' 1024 columns, fewer rows than a statistics slab (8, 20), next
# to m <= n matrices.
COLPATH_SHAPES = [(1000, 332), (2049, 256), (130, 20), (5000, 516), (300, 8), (64, 64), (256, 1024),
                 (20000, 132)]


@pytest.mark.parametrize("grad_dtype", ["bf16", "f32"])
def test_rownorm_column_path_aligned_and_not(grad_dtype):
    """The m > n matrices take the three column kernels beside the row kernels, with W
    16-byte aligned (vector loads) or one float past the boundary (element by element).
    Within 1e-5 of the oracle over two steps in a row."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    inputs = host_inputs(COLPATH_SHAPES, grad_dtype, base_seed=34)
    plan = lib.MuonPlan(COLPATH_SHAPES, grad_dtype)
    row_launches = len({lib_row_class(n) for m, n in COLPATH_SHAPES if m <= n})
    for aligned in (True, False):
        W = []
        for w, _, _ in inputs:
            if aligned:
                W.append(w.cuda())
            else:   # every W one float past a 16-byte boundary
                buf = torch.empty(w.numel() + 1, device="cuda")
                v = buf[1:].view(w.shape)
                v.copy_(w.cuda())
                W.append(v)
        G = [x[1].cuda() for x in inputs]
        M = [x[2].cuda() for x in inputs]
        w_ref = [x[0].double().numpy() for x in inputs]
        m_ref = [x[2].double().numpy() for x in inputs]
        for t in range(2):
            plan.rownorm_step(W, G, M, LR, WD, MU, 1e-8)
            plan.sync()
            assert plan.info()["launches_last_step"] == row_launches + 3
            for i in range(len(COLPATH_SHAPES)):
                w_ref[i], m_ref[i], _ = R.muon_step(w_ref[i], inputs[i][1].double().numpy(), m_ref[i], LR, WD, MU,
                                                    0, "rownorm", 1e-8)
                assert rel(M[i].cpu().numpy(), m_ref[i]) <= TOL_FP32, (COLPATH_SHAPES[i], aligned, t)
                assert rel(W[i].cpu().numpy(), w_ref[i]) <= TOL_FP32, (COLPATH_SHAPES[i], aligned, t)
    plan.close()


def lib_row_class(n):
    """Launch class of a RowNorm row of n elements (rows up to 2048, 4096, longer)."""
    return 0 if n <= 2048 else (1 if n <= 4096 else 2)


def test_rownorm_eps_floor():
    """Rows whose norm is below eps are divided by eps, not normalised."""
    import torch
    shapes = [(8, 32), (32, 8)]
    inputs = [(w, g * 1e-9, m * 0) for w, g, m in host_inputs(shapes, "f32", 32)]
    eps = 1e-3
    res = run_step(shapes, "f32", inputs=inputs, mode="rownorm", eps=eps, keep_update=False)
    for i in range(2):
        e = check_rownorm_matrix(res, i, eps=eps)
        assert e["m"] <= TOL_FP32 and e["w"] <= TOL_FP32, e


def test_periodic_rownorm_schedule_matches_oracle():
    """K = 4 over 8 steps (NS at t = 0 and 4), fresh gradients each step."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    from workloads import gen_tensor, seed_of, G_STD
    shapes = [(96, 320), (320, 96)]
    inputs = host_inputs(shapes, "bf16", 33)
    plan = lib.MuonPlan(shapes, "bf16")
    sched = lib.PeriodicRowNormMuon(plan, k=4)
    W = [x[0].cuda() for x in inputs]
    M = [x[2].cuda() for x in inputs]
    w_ref = [x[0].double().numpy() for x in inputs]
    m_ref = [x[2].double().numpy() for x in inputs]
    for t in range(8):
        grads = [gen_tensor(s, G_STD, seed_of(33, t, i, "G"), dtype="bf16") for i, s in enumerate(shapes)]
        mode = sched.step(W, [g.cuda() for g in grads], M, LR, WD)
        assert mode == R.schedule_mode(t, 4)
        for i in range(2):
            w_ref[i], m_ref[i], _ = R.muon_step(w_ref[i], grads[i].double().numpy(), m_ref[i], LR, WD, MU,
                                                5, mode, 1e-8)
    plan.sync()
    for i in range(2):
        assert rel(M[i].cpu().numpy(), m_ref[i]) <= TOL_FP32
        # two NS steps with O at <= 2e-2 each: W within lr * s * 2e-2 * ||O|| per NS step
        bound = 2 * LR * R.update_scale(*shapes[i]) * TOL_O * np.sqrt(min(shapes[i])) / np.linalg.norm(w_ref[i])
        assert rel(W[i].cpu().numpy(), w_ref[i]) <= bound + 1e-5


# --------------------------------------------------------------- host validation through the ABI
def test_invalid_arguments_are_rejected_without_touching_buffers():
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(32, 64)]
    inp = host_inputs(shapes, "bf16", 41)
    plan = lib.MuonPlan(shapes, "bf16")
    W, G, M = inp[0][0].cuda(), inp[0][1].cuda(), inp[0][2].cuda()
    W0, M0 = W.clone(), M.clone()
    with pytest.raises(lib.MuonError) as ei:
        plan.step([W], [G], [M], LR, WD, 1.0)
    assert ei.value.code == lib.MUON_ERR_INVALID_ARG
    with pytest.raises(lib.MuonError):
        plan.step([W], [G], [M], LR, WD, MU, ns_steps=6)     # beyond the Gram recursion's stable range
    with pytest.raises(lib.MuonError):
        plan.step([W], [G], [M], LR, WD, MU, ns_steps=-1)
    with pytest.raises(lib.MuonError):
        plan.step([W], [G], [M], float("nan"), WD, MU)
    with pytest.raises(lib.MuonError):
        plan.rownorm_step([W], [G], [M], LR, WD, MU, eps=0.0)
    with pytest.raises(lib.MuonError):      # params aliasing momentum
        plan.step([W], [G], [W], LR, WD, MU)
    with pytest.raises(ValueError):
        plan.step([W], [G.float()], [M], LR, WD, MU)
    torch.cuda.synchronize()
    assert torch.equal(W, W0) and torch.equal(M, M0)
    plan.sync()


@pytest.mark.parametrize("chain_clusters", [-1, 6])
def test_stage_times_split_fused_and_gemm_stages(chain_clusters):
    """muon_stage_times: six stages; the fused r <= 128 step has its own stage and
    its matrices are left out of the GEMM stages' algorithmic FLOPs.  Run in
    sequence (chain_clusters -1) the stages of NS steps add up to the step time;
    overlapped (6 CTA pairs for the batched products) they run beside the fused one."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    from workloads import gen_tensor
    shapes = [(128, 1000), (300, 700), (700, 300), (64, 64)]
    W = [gen_tensor(s, 0.02, 7 + i, "cuda") for i, s in enumerate(shapes)]
    G = [gen_tensor(s, 1e-3, 17 + i, "cuda") for i, s in enumerate(shapes)]
    M = [gen_tensor(s, 1e-3, 27 + i, "cuda") for i, s in enumerate(shapes)]
    plan = lib.MuonPlan(shapes, "f32", timing=True, chain_clusters=chain_clusters)
    plan.step(W, G, M, LR, WD, MU, 5, "ns")
    plan.sync()
    plan.stage_times()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(3):
        plan.step(W, G, M, LR, WD, MU, 5, "ns")
    ev1.record()
    plan.sync()
    torch.cuda.synchronize()
    ms, fl = plan.stage_times()
    assert len(ms) == 6 and all(x >= 0 for x in ms)
    assert ms[4] == 0.0                      # no RowNorm step ran
    assert all(ms[k] > 0 for k in (0, 1, 2, 3, 5))
    total = ev0.elapsed_time(ev1)
    batched = ms[1] + ms[2] + ms[3]
    span = ms[0] + (ms[5] + batched if chain_clusters < 0 else max(ms[5], batched))
    assert 0.7 * total <= span <= 1.05 * total, (ms, total)
    r, c = 300, 700                          # the two non-fused matrices (one per orientation)
    assert fl[0] == pytest.approx(3 * 2 * r * r * c)
    assert fl[1] == pytest.approx(3 * 2 * 17 * r ** 3)
    assert fl[2] == pytest.approx(3 * 2 * 2 * r * r * c)
    plan.close()


def test_overlapped_fused_and_batched_match_sequential_bitwise():
    """The fused and batched matrices of one plan run side by side on two streams
    (automatic split) or one after the other (chain_clusters -1); every tile's
    arithmetic is the same either way, so W, M and O agree bit for bit."""
    import torch
    shapes = [(128, 1000), (100, 3000), (300, 700), (700, 300), (64, 64), (520, 2100)]
    inputs = host_inputs(shapes, "bf16", base_seed=77)
    outs = []
    for cc in (0, -1, 5):
        res = run_step(shapes, "bf16", inputs=inputs, chain_clusters=cc)
        outs.append(res)
    for res in outs[1:]:
        for i in range(len(shapes)):
            assert torch.equal(res["W"][i], outs[0]["W"][i]), i
            assert torch.equal(res["M"][i], outs[0]["M"][i]), i
            assert torch.equal(res["O"][i], outs[0]["O"][i]), i


def test_bounded_wait_expiry_is_reported_and_plan_recovers():
    """Failure detection without a fault: a device wait that nothing completes gives
    up after its limit, muon_sync reports MUON_ERR_TIMEOUT once, and the same plan
    then steps correctly (checked against the oracle)."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(256, 1024), (100, 700)]
    inputs = host_inputs(shapes, "f32", base_seed=91)
    plan = lib.MuonPlan(shapes, "f32", keep_update=True)
    plan.debug_wait_timeout(500)
    with pytest.raises(lib.MuonError) as ei:
        plan.sync()
    assert ei.value.code == lib.MUON_ERR_TIMEOUT
    plan.sync()                               # the status word was cleared
    res = run_step(shapes, "f32", inputs=inputs, plan=plan)
    for i in range(len(shapes)):
        assert_ns(res, i)
    with pytest.raises(lib.MuonError):
        plan.debug_wait_timeout(0)            # limit outside [1, 1e6] us: refused on the host
    plan.close()


@pytest.mark.parametrize("mode", ["ns", "rownorm"])
def test_check_finite_reports_a_nan_gradient(mode):
    """opts.check_finite: a NaN in one gradient makes that matrix's input norm
    non-finite; muon_sync reports MUON_ERR_NONFINITE once, the other matrices are
    updated as usual, and the next step with finite gradients syncs clean.  Without the
    option the same step reports nothing.  Covers the Frobenius norm of NS steps (fused,
    fp32 and batched matrices) and the row and column norms of RowNorm steps."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(256, 1024), (1024, 256), (100, 700), (96, 96)]
    for bad in range(len(shapes)):
        inputs = host_inputs(shapes, "bf16", base_seed=92)
        g = inputs[bad][1].clone()
        g[3, 5] = float("nan")
        inputs[bad] = (inputs[bad][0], g, inputs[bad][2])
        for check in (True, False):
            plan = lib.MuonPlan(shapes, "bf16", check_finite=check)
            W = [x[0].cuda() for x in inputs]
            G = [x[1].cuda() for x in inputs]
            M = [x[2].cuda() for x in inputs]
            if mode == "ns":
                plan.step(W, G, M, LR, WD, MU, 5, "ns")
            else:
                plan.rownorm_step(W, G, M, LR, WD, MU, 1e-8)
            if check:
                with pytest.raises(lib.MuonError) as ei:
                    plan.sync()
                assert ei.value.code == lib.MUON_ERR_NONFINITE, (bad, mode)
            plan.sync()   # reported once (or, unchecked, never)
            for i in range(len(shapes)):
                if i != bad:
                    assert bool(torch.isfinite(W[i]).all()), (bad, i)
            clean = [x[1].cuda() for x in host_inputs(shapes, "bf16", base_seed=93)]
            M = [x[2].cuda() for x in host_inputs(shapes, "bf16", base_seed=93)]
            plan.step(W, clean, M, LR, WD, MU, 5, mode)
            plan.sync()
            plan.close()


def test_workspace_cap_runs_the_step_in_chunks_bitwise():
    """opts.workspace_bytes: the NS step runs chunk by chunk on one shared region of
    X0 and r x r buffers; every matrix gets bit for bit the update of the uncapped
    plan, two steps in a row, and a cap below one matrix's needs is refused."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(520, 2100), (2100, 520), (384, 384), (130, 300), (300, 130), (128, 1000), (64, 64),
              (256, 1024)] * 2
    inputs = host_inputs(shapes, "bf16", base_seed=55)
    ref = run_step(shapes, "bf16", inputs=inputs)
    full = ref["plan"].info()
    ref2 = run_step(shapes, "bf16", inputs=[(w, g, m) for w, (_, g, _), m in
                                            zip(ref["W"], inputs, ref["M"])], plan=ref["plan"])
    chunked = 0
    for frac in (0.7, 0.5, 0.35):
        cap = int(full["workspace_bytes"] * frac)
        try:
            res = run_step(shapes, "bf16", inputs=inputs, workspace_bytes=cap)
        except lib.MuonError as e:
            assert e.code == lib.MUON_ERR_OOM
            continue
        info = res["plan"].info()
        assert info["workspace_bytes"] <= cap
        chunked += info["n_buckets"] > full["n_buckets"]
        for i in range(len(shapes)):
            assert torch.equal(res["W"][i], ref["W"][i]), (frac, i)
            assert torch.equal(res["M"][i], ref["M"][i]), (frac, i)
            assert torch.equal(res["O"][i], ref["O"][i]), (frac, i)
        res2 = run_step(shapes, "bf16", inputs=[(w, g, m) for w, (_, g, _), m in
                                                zip(res["W"], inputs, res["M"])], plan=res["plan"])
        for i in range(len(shapes)):
            assert torch.equal(res2["W"][i], ref2["W"][i]), (frac, i)
        res["plan"].close()
    assert chunked >= 1
    with pytest.raises(lib.MuonError) as ei:
        lib.MuonPlan(shapes, "bf16", workspace_bytes=1 << 20)
    assert ei.value.code == lib.MUON_ERR_OOM
    ref["plan"].close()


# ---- NS coefficient and step variants (muon_step_ex)
VARIANT_SHAPES = [(128, 1000), (100, 700), (300, 130), (520, 2100), (256, 1024)]


def check_ns_variant(res, i, steps, coeffs, tol):
    """M and W-given-O to 1e-5, O against the oracle's direct NS with these steps and coefficients."""
    w, g, m = (t.double().numpy() for t in res["inputs"][i])
    _, m_ref, o_ref = R.muon_step(w, g, m, LR, WD, MU, steps, "ns", 1e-8, coeffs)
    o = res["O"][i].double().numpy()
    assert rel(res["M"][i].numpy(), m_ref) <= TOL_FP32, i
    mm, nn = o.shape
    assert rel(res["W"][i].numpy(), R.apply_update(w, o, LR, WD, R.update_scale(mm, nn))) <= TOL_FP32, i
    e = rel(o, o_ref)
    assert e <= tol, (i, res["inputs"][i][0].shape, e)
    return e


@pytest.mark.parametrize("coeffs", [(1.5, -0.5, 0.0), (2.0, -1.5, 0.5)])
def test_custom_coefficients_match_oracle(coeffs):
    """Cubic NS and another quintic through muon_step_ex, on the fused r <= 128 kernel
    and the CTA-pair path of one plan."""
    res = run_step(VARIANT_SHAPES, "bf16", base_seed=61, coeffs=coeffs)
    for i in range(len(VARIANT_SHAPES)):
        check_ns_variant(res, i, 5, coeffs, TOL_O)


@pytest.mark.parametrize("steps,restart", [(10, 0), (7, 3), (4, 1)])
def test_restarted_segments_match_oracle(steps, restart):
    """ns_steps beyond one segment (10 = 5 + 5, 7 = 3 + 3 + 1) and the direct form
    (restart 1): the iterate is formed between segments and the next Gram matrix
    recomputed from it."""
    res = run_step(VARIANT_SHAPES, "bf16", base_seed=62, ns_steps=steps, restart=restart, max_ns_steps=10)
    for i in range(len(VARIANT_SHAPES)):
        check_ns_variant(res, i, steps, R.NS_COEFFS, TOL_O)


def test_restart_every_step_on_ill_conditioned_input():
    """Singular values spread from 1 to 1e-4 on the plain recipe (precision -1): the Gram
    form carries fp16 rounding of G into the small singular directions through Q
    (measured 0.17 on GB300); the direct form (restart 1) recomputes X X^T from the
    iterate every step and cuts the error to less than half (measured 0.073).  It stays
    above the 2e-2 bar: the iterates are bf16 (X0 from the momentum pass, X' between
    steps), whose rounding the small singular directions cannot carry; precision 2
    (test_split_level_2_on_an_ill_conditioned_input) removes that limit.  The bounds
    pinned here are the measured values plus 30 %."""
    import torch
    rng = np.random.default_rng(7)
    r, c = 256, 1024
    a, _ = np.linalg.qr(rng.standard_normal((r, r)))
    b, _ = np.linalg.qr(rng.standard_normal((c, r)))
    u = (a * np.logspace(0, -4, r)) @ b.T * 1e-3
    g = torch.from_numpy(u / (1 + MU)).float()            # with M = 0: U = (1 + mu) G
    w = torch.from_numpy(rng.standard_normal((r, c)) * 0.02).float()
    inputs = [(w, g, torch.zeros(r, c))]
    errs = {}
    for restart, bound in ((5, 0.22), (1, 0.095)):
        res = run_step([(r, c)], "f32", inputs=inputs, restart=restart, max_ns_steps=5, precision=-1)
        errs[restart] = check_ns_variant(res, 0, 5, R.NS_COEFFS, bound)
    assert errs[1] < 0.6 * errs[5], errs


def test_step_ex_argument_checks():
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(64, 256), (300, 700)]
    W = [torch.zeros(s, device="cuda") for s in shapes]
    G = [torch.zeros(s, device="cuda") for s in shapes]
    M = [torch.zeros(s, device="cuda") for s in shapes]
    plan = lib.MuonPlan(shapes, "f32")
    cases = [(dict(ns_steps=6), lib.MUON_ERR_INVALID_ARG),              # beyond one segment, no restarts
             (dict(ns_steps=5, restart=2), lib.MUON_ERR_UNSUPPORTED),   # needs max_ns_steps
             (dict(ns_steps=5, restart=6), lib.MUON_ERR_INVALID_ARG),
             (dict(ns_steps=5, coeffs=(float("nan"), 0.0, 0.0)), lib.MUON_ERR_INVALID_ARG)]
    for kw, code in cases:
        with pytest.raises(lib.MuonError) as ei:
            plan.step(W, G, M, LR, WD, MU, kw.pop("ns_steps"), "ns", **kw)
        assert ei.value.code == code, kw
    plan.close()
    with pytest.raises(lib.MuonError) as ei:
        lib.MuonPlan(shapes, "f32", max_ns_steps=101)
    assert ei.value.code == lib.MUON_ERR_INVALID_ARG


HOST_SHAPES = [(128, 3584)] * 6 + [(300, 65), (7, 13)] + [(520, 200)] * 3 + [(200, 520)] * 2 + [(1024, 256)]


def _two_steps_on_device(plan, shapes, grads, mode):
    """Reference for muon_step_host: the same two steps with the gradients already on the device."""
    import torch
    inp = host_inputs(shapes, "bf16", 41)
    W = [w.cuda() for w, _, _ in inp]
    M = [m.cuda() for _, _, m in inp]
    G = [torch.empty_like(g, device="cuda") for g in grads[0]]
    for step_grads in grads:
        for gd, gh in zip(G, step_grads):
            gd.copy_(gh)
        if mode == "ns":
            plan.step(W, G, M, LR, WD, MU, 5, "ns")
        else:
            plan.rownorm_step(W, G, M, LR, WD, MU)
    plan.sync()
    return [w.cpu() for w in W], [m.cpu() for m in M]


@pytest.mark.parametrize("mode", ["ns", "rownorm"])
def test_step_host_overlapped_copies_match_device_step(mode):
    """muon_step_host on a plan split into chunks (gradients copied in and params copied
    back on the plan's copy streams, overlapped with the compute) gives bitwise the
    results of the same two steps run on device buffers by an unchunked plan; the host
    copies of the params equal the device params, and the second step's copies in wait
    for the first step's reads of the gradient buffers."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = HOST_SHAPES
    grads = [[g for _, g, _ in host_inputs(shapes, "bf16", 41, step=t)] for t in (0, 1)]
    ref_plan = lib.MuonPlan(shapes, "bf16")
    W_ref, M_ref = _two_steps_on_device(ref_plan, shapes, grads, mode)
    ref_plan.close()

    plan = lib.MuonPlan(shapes, "bf16", chunks=4)
    assert plan.info()["n_chunks"] >= 3
    inp = host_inputs(shapes, "bf16", 41)
    W = [w.cuda() for w, _, _ in inp]
    M = [m.cuda() for _, _, m in inp]
    G = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    gh = [[g.pin_memory() for g in step_grads] for step_grads in grads]
    wh = [torch.empty(s, dtype=torch.float32).pin_memory() for s in shapes]
    for t in range(2):
        plan.step_host(W, G, M, gh[t], wh, LR, WD, MU, 5, mode)
    torch.cuda.current_stream().synchronize()
    plan.sync()
    for i in range(len(shapes)):
        assert torch.equal(W[i].cpu(), W_ref[i]), (mode, i, shapes[i])
        assert torch.equal(M[i].cpu(), M_ref[i]), (mode, i, shapes[i])
        assert torch.equal(wh[i], W_ref[i]), (mode, i, shapes[i])
        assert torch.equal(G[i].cpu(), grads[1][i]), (mode, i, shapes[i])
    plan.close()


def test_step_host_without_copy_back_and_argument_checks():
    import ctypes
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = HOST_SHAPES
    grads = [[g for _, g, _ in host_inputs(shapes, "bf16", 41, step=0)]]
    ref_plan = lib.MuonPlan(shapes, "bf16")
    W_ref, M_ref = _two_steps_on_device(ref_plan, shapes, grads, "ns")
    ref_plan.close()
    plan = lib.MuonPlan(shapes, "bf16")   # one chunk
    inp = host_inputs(shapes, "bf16", 41)
    W = [w.cuda() for w, _, _ in inp]
    M = [m.cuda() for _, _, m in inp]
    G = [torch.zeros(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
    w0 = [w.clone() for w in W]
    # a null host gradient pointer: rejected before anything is enqueued
    w, g, m = plan._pointers(W, G, M)
    gh = (ctypes.c_void_p * len(shapes))(*([grads[0][0].data_ptr()] + [None] * (len(shapes) - 1)))
    code = plan.lib.muon_step_host(plan.handle, w, g, m, gh, None, LR, WD, MU, 5, lib.MUON_MODE_NS, None)
    assert code == lib.MUON_ERR_INVALID_ARG
    gh = (ctypes.c_void_p * len(shapes))(*[t.data_ptr() for t in grads[0]])
    code = plan.lib.muon_step_host(plan.handle, w, g, m, gh, None, LR, WD, MU, 6, lib.MUON_MODE_NS, None)
    assert code == lib.MUON_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(W, w0)) and all(int(t.abs().sum()) == 0 for t in G)
    plan.step_host(W, G, M, grads[0], None, LR, WD, MU, 5, "ns")   # pageable host memory
    torch.cuda.synchronize()
    plan.sync()
    for i in range(len(shapes)):
        assert torch.equal(W[i].cpu(), W_ref[i]) and torch.equal(M[i].cpu(), M_ref[i]), i
    plan.close()


@pytest.mark.parametrize("shapes", [
    [(512, 1024), (1024, 2048), (2048, 1024), (768, 1536), (512, 4096)],   # r, c multiples of 64: lower triangle
    [(512, 1024), (700, 900), (128, 3584)],                              # a ragged bucket: stored whole
])
def test_lower_triangle_storage_matches_whole_storage_bitwise(shapes):
    """Symmetric r x r results stored as their lower triangle (the products read the
    blocks above the diagonal tile from the mirror position through 4-D maps) give
    bitwise the results of whole storage: the same MMAs on the same operand values."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    lplan = lib.MuonPlan(shapes, "bf16", keep_update=True)
    aligned = all(min(m, n) % 64 == 0 and max(m, n) % 64 == 0 for m, n in shapes if min(m, n) > 128)
    assert lplan.info()["lower_chunks"] == (1 if aligned else 0)
    low = run_step(shapes, "bf16", base_seed=51, plan=lplan)
    plan = lib.MuonPlan(shapes, "bf16", keep_update=True, full_symmetric=True)
    assert plan.info()["lower_chunks"] == 0
    whole = run_step(shapes, "bf16", inputs=low["inputs"], plan=plan)
    for i in range(len(shapes)):
        assert torch_equal(low["W"][i], whole["W"][i]), shapes[i]
        assert torch_equal(low["O"][i], whole["O"][i]), shapes[i]
        assert_ns(low, i)
    # the workspace copies rebuild the upper part: same G, P, Q as whole storage
    for i, (m, n) in enumerate(shapes):
        if min(m, n) > 128:
            for which in (1, 2, 3, 5, 6, 7):
                assert torch_equal(lplan.debug_workspace(i, which), plan.debug_workspace(i, which)), (i, which)
    plan.close()
    lplan.close()


def torch_equal(a, b):
    import torch
    return torch.equal(a, b)


def test_plan_tune_keeps_results_bitwise():
    """muon_plan_tune times the speed-only launch choices (CTA pairs beside the fused kernel,
    clusters of two pairs for the final product) and keeps the fastest; a step of the tuned
    plan gives bitwise the results of the untuned plan."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(128, 3584)] * 64 + [(3584, 512)] * 4 + [(1024, 2048)] * 2
    inputs = host_inputs(shapes, "bf16", 71)
    ref = run_step(shapes, "bf16", inputs=inputs)
    plan = lib.MuonPlan(shapes, "bf16", keep_update=True)
    W = [w.cuda() for w, _, _ in inputs]
    G = [g.cuda() for _, g, _ in inputs]
    M = [m.cuda() for _, _, m in inputs]
    ms = plan.tune(W, G, M, LR, WD, MU, reps=2)
    info = plan.info()
    assert ms > 0 and info["tuned_candidates"] >= 2, (ms, info)
    res = run_step(shapes, "bf16", inputs=inputs, plan=plan)
    for i in range(len(shapes)):
        assert torch.equal(res["W"][i], ref["W"][i]), (i, info)
        assert torch.equal(res["M"][i], ref["M"][i]), (i, info)
        assert torch.equal(res["O"][i], ref["O"][i]), (i, info)
    with pytest.raises(lib.MuonError):
        plan.tune(W, G, M, LR, WD, MU, reps=0)
    plan.close()


@pytest.mark.parametrize("ns_steps,restart", [(0, 0), (1, 0), (2, 0), (7, 3), (4, 1)])
def test_lower_triangle_storage_other_steps_and_restarts(ns_steps, restart):
    """Lower-triangle storage with J = 0 (identity Q), 1 (P and Q stored whole by the
    per-thread epilogue), 2, and restarted segments (the second X buffer's 4-D maps, X'
    formed between segments): bitwise the results of whole storage, and the oracle's."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(192, 576), (576, 192), (256, 1024)]
    mx = 10 if restart else 0
    lplan = lib.MuonPlan(shapes, "bf16", keep_update=True, max_ns_steps=mx)
    assert lplan.info()["lower_chunks"] == 1
    low = run_step(shapes, "bf16", base_seed=81, ns_steps=ns_steps, restart=restart, plan=lplan)
    wplan = lib.MuonPlan(shapes, "bf16", keep_update=True, max_ns_steps=mx, full_symmetric=True)
    whole = run_step(shapes, "bf16", inputs=low["inputs"], ns_steps=ns_steps, restart=restart, plan=wplan)
    for i in range(len(shapes)):
        assert torch_equal(low["W"][i], whole["W"][i]), (i, ns_steps, restart)
        assert torch_equal(low["O"][i], whole["O"][i]), (i, ns_steps, restart)
        assert_ns(low, i, ns_steps=ns_steps)
    lplan.close()
    wplan.close()


def test_plan_allocates_what_host_sizing_reports():
    """muon_plan_workspace_size (host only) and a real plan agree on the workspace
    bytes, buckets and chunks, with and without caps, chunks, restarts and the O copy."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    layer = [(3584, 3584), (512, 3584), (512, 3584), (3584, 3584), (18944, 3584), (18944, 3584), (3584, 18944)]
    mixed = [(300, 1000), (1000, 300), (64, 64), (129, 4096), (4096, 256)] * 3
    cases = [(layer, {}), (layer, {"chunks": 3}), (layer, {"max_ns_steps": 10}),
             (mixed, {}), (mixed, {"keep_update": True}), (mixed, {"generic_small": True, "chunks": 4})]
    full = lib.plan_workspace_size(layer)["workspace_bytes"]
    cases.append((layer, {"workspace_bytes": full - 1}))
    for shapes, opts in cases:
        est = lib.plan_workspace_size(shapes, "bf16", **opts)
        plan = lib.MuonPlan(shapes, "bf16", **opts)
        info = plan.info()
        plan.close()
        got = {"workspace_bytes": info["workspace_bytes"], "n_buckets": info["n_buckets"],
               "n_chunks": info["n_chunks"]}
        assert got == est, (opts, got, est)
    assert lib.plan_workspace_size(layer, workspace_bytes=full - 1)["n_chunks"] >= 2


LONGEST = [(1, 1 << 20), (1 << 20, 8), (1 << 20, 136)]


@pytest.mark.parametrize("mode", ["ns", "rownorm"])
def test_longest_side_the_library_accepts(mode):
    """Long side 2^20, the per-dimension limit: a row vector and a thin transposed matrix
    on the fused kernel, and r = 136 on the CTA-pair kernel (one ragged 256 x 256 pair
    tile whose SYRK runs 2^14 k-blocks)."""
    res = run_step(LONGEST, "bf16", base_seed=77, mode=mode)
    for i in range(len(LONGEST)):
        if mode == "ns":
            assert_ns(res, i)
        else:
            e = check_rownorm_matrix(res, i)
            assert e["m"] <= TOL_FP32 and e["w"] <= TOL_FP32, (i, e)


@pytest.mark.parametrize("shapes,lower", [
    (RAGGED, False),
    ([(640, 1280), (1280, 640), (256, 1024), (128, 2048), (2048, 64)], True),
], ids=["ragged", "lower_triangle"])
def test_steps_write_nothing_outside_the_callers_buffers(shapes, lower):
    """Every W, G and M is a view into a larger allocation, 4096 elements of guard on each
    side (the views stay 256-byte aligned, so the kernels take their usual paths).  After
    an NS step and a RowNorm step every guard is bit-identical and G is untouched."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    guard = 4096
    inputs = host_inputs(shapes, "bf16", base_seed=91)
    bufs, views = [], {"W": [], "G": [], "M": []}
    for w, g, m in inputs:
        for name, t in (("W", w), ("G", g), ("M", m)):
            n = t.numel()
            buf = torch.randn(n + 2 * guard, device="cuda").to(t.dtype)
            view = buf[guard:guard + n].view(t.shape)
            view.copy_(t.cuda())
            assert view.is_contiguous() and view.data_ptr() % 256 == buf.data_ptr() % 256
            bufs.append((buf, n, buf.clone()))
            views[name].append(view)
    g_before = [g.clone() for g in views["G"]]
    plan = lib.MuonPlan(shapes, "bf16")
    plan.step(views["W"], views["G"], views["M"], LR, WD, MU, 5, "ns")
    plan.rownorm_step(views["W"], views["G"], views["M"], LR, WD, MU, 1e-8)
    plan.sync()
    for buf, n, ref in bufs:
        assert torch.equal(buf[:guard], ref[:guard]) and torch.equal(buf[guard + n:], ref[guard + n:])
    for g, g0 in zip(views["G"], g_before):
        assert torch.equal(g, g0)
    if lower:
        assert plan.info()["lower_chunks"] == 1


def test_resume_from_saved_state_is_bitwise():
    """Eight periodic RowNorm Muon steps (K = 4, fresh gradients each step) run straight
    equal, bitwise, four steps, a save of W, M and the schedule to host memory, a new plan
    restored from the save, and four more steps.  The optimizer's state is the momentum
    and the step index; the plan keeps nothing else between steps."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(300, 1000), (1000, 300), (128, 512), (640, 1280), (64, 4096)]
    base = host_inputs(shapes, "bf16", base_seed=55)
    grads = [[g for _, g, _ in host_inputs(shapes, "bf16", base_seed=55, step=t)] for t in range(8)]

    def run(steps, W, M, state=None):
        plan = lib.MuonPlan(shapes, "bf16")
        sched = lib.PeriodicRowNormMuon(plan, k=4)
        if state is not None:
            sched.load_state_dict(state)
        for t in steps:
            assert sched.t == t
            sched.step(W, [g.cuda() for g in grads[t]], M, LR, WD)
        plan.sync()
        out = sched.state_dict()
        plan.close()
        return out

    W1 = [w.cuda() for w, _, _ in base]
    M1 = [m.cuda() for _, _, m in base]
    run(range(8), W1, M1)
    W2 = [w.cuda() for w, _, _ in base]
    M2 = [m.cuda() for _, _, m in base]
    state = run(range(4), W2, M2)
    saved = ([w.cpu() for w in W2], [m.cpu() for m in M2], dict(state))
    del W2, M2
    W3 = [w.cuda() for w in saved[0]]
    M3 = [m.cuda() for m in saved[1]]
    run(range(4, 8), W3, M3, saved[2])
    for i in range(len(shapes)):
        assert torch.equal(W1[i], W3[i]), ("W", i)
        assert torch.equal(M1[i], M3[i]), ("M", i)


def test_distributed_muon_on_one_rank_is_the_plan_step_bitwise():
    """DistributedMuon without a process group (one rank owns every matrix): its step is
    the plan's step, bitwise, in both modes; with allocate_params the parameters are views
    into one flat buffer."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(300, 700), (700, 300), (128, 512), (96, 96)]
    inputs = host_inputs(shapes, "bf16", base_seed=71)
    opt = lib.DistributedMuon(shapes, "bf16")
    assert opt.world == 1 and opt.owned == list(range(len(shapes)))
    W1 = opt.allocate_params("cuda")
    for w, (w0, _, _) in zip(W1, inputs):
        w.copy_(w0.cuda())
    M1 = [m.cuda() for _, _, m in inputs]
    plan = lib.MuonPlan(shapes, "bf16")
    W2 = [w.cuda() for w, _, _ in inputs]
    M2 = [m.cuda() for _, _, m in inputs]
    for mode in ("ns", "rownorm", "ns"):
        G = [g.cuda() for _, g, _ in inputs]
        opt.step(W1, G, M1, LR, WD, MU, 5, mode)
        if mode == "ns":
            plan.step(W2, G, M2, LR, WD, MU, 5, "ns")
        else:
            plan.rownorm_step(W2, G, M2, LR, WD, MU, 1e-8)
    opt.sync()
    plan.sync()
    for i in range(len(shapes)):
        assert torch.equal(W1[i], W2[i]) and torch.equal(M1[i], M2[i]), i
    opt.close()
    plan.close()


# --------------------------------------------------------------- split precision (opts.precision)
NEAR_SQUARE = [(256, 256), (384, 384), (512, 512), (200, 210), (300, 256), (576, 640)]


def test_near_square_batched_buckets_split_by_default():
    """Nearly square batched buckets (r > 128) carry the r x r recursion and Q in two parts
    (precision 0 picks level 1 for them): O within the bar with margin (emulated 3-4e-3;
    the plain recipe measured 2.1e-2 on 256 x 256), next to rectangular buckets that stay
    plain in the same plan."""
    shapes = NEAR_SQUARE + [(300, 700), (700, 300)]
    res = run_step(shapes, "bf16", base_seed=33)
    assert res["plan"].info()["split_buckets"] == len(NEAR_SQUARE)
    for i in range(len(NEAR_SQUARE)):
        e = assert_ns(res, i)
        assert e["o"] <= 1e-2, (shapes[i], e)
    for i in range(len(NEAR_SQUARE), len(shapes)):
        assert_ns(res, i)
    plain = run_step(shapes, "bf16", base_seed=33, precision=-1)
    assert plain["plan"].info()["split_buckets"] == 0


@pytest.mark.parametrize("ns_steps", [0, 1, 2, 5])
def test_small_squares_on_the_batched_split_path(ns_steps):
    """r <= 128 squares on the batched products (generic_small, small_fp32 = -1) with
    precision 1: the one-SM kernel's split passes meet the bar at every step count."""
    shapes = [(64, 64), (96, 96), (128, 128), (100, 100), (128, 3584)]
    res = run_step(shapes, "bf16", base_seed=34, ns_steps=ns_steps, generic_small=True, small_fp32=-1,
                   precision=1)
    assert res["plan"].info()["split_buckets"] == len(shapes)
    for i in range(len(shapes)):
        e = assert_ns(res, i, ns_steps=ns_steps)
        assert e["o"] <= 1e-2, (shapes[i], e)


@pytest.mark.parametrize("precision", [1, 2])
def test_split_levels_on_the_ragged_plan(precision):
    """Every batched bucket of the ragged plan split (level 1, or 2 with X0 in two parts as
    well): both orientations, ragged tails, the one-SM and the CTA-pair kernels."""
    res = run_step(RAGGED, "bf16", base_seed=21, precision=precision)
    for i in range(len(RAGGED)):
        e = assert_ns(res, i)
        assert e["o"] <= 1e-2, (RAGGED[i], e)


def test_split_level_2_on_an_ill_conditioned_input():
    """Singular values spread from 1 to 1e-4 (as in the restart test): the plain recipe
    measured 0.17 (Gram form) and 0.073 (restart every step); with X0, the recursion and
    Q all in two parts the error falls below the 2e-2 bar (emulated: 9e-5 with fp32 X0,
    4.8e-2 with a one-part bf16 X0)."""
    import torch
    rng = np.random.default_rng(7)
    r, c = 256, 1024
    a, _ = np.linalg.qr(rng.standard_normal((r, r)))
    b, _ = np.linalg.qr(rng.standard_normal((c, r)))
    u = (a * np.logspace(0, -4, r)) @ b.T * 1e-3
    g = torch.from_numpy(u / (1 + MU)).float()
    w = torch.from_numpy(rng.standard_normal((r, c)) * 0.02).float()
    res = run_step([(r, c)], "f32", inputs=[(w, g, torch.zeros(r, c))], precision=2)
    e = assert_ns(res, 0)
    assert e["o"] <= 2e-2, e


@pytest.mark.parametrize("precision", [1, 2])
def test_split_levels_with_restarted_segments(precision):
    """Ten steps in two restarted segments: the iterate between them is written in two
    parts at level 2 and read back by the next SYRK."""
    res = run_step(VARIANT_SHAPES, "bf16", base_seed=62, ns_steps=10, max_ns_steps=10, precision=precision)
    for i in range(len(VARIANT_SHAPES)):
        check_ns_variant(res, i, 10, R.NS_COEFFS, TOL_O)


def test_dim0_shard_rownorm_matches_the_full_matrix():
    """RowNorm over dim-0 shards (opts.full_rows) on one GPU: every matrix split into two
    row blocks that one plan holds as separate shards; the column sums of the two blocks
    are added on the device between the two shard calls (what an all-reduce across ranks
    does), and the blocks together must equal the oracle's RowNorm step on the full
    matrix (M and W at 1e-5).  Covers spanning (m > n) and complete (m <= n) rows."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    from workloads import gen_tensor, seed_of
    full = [(1000, 333), (333, 1000), (12288, 2048), (256, 1024), (2048, 2048), (130, 7)]
    shards, full_rows, parts = [], [], []
    for i, (m, n) in enumerate(full):
        k = (m // 3) // 8 * 8 + 5                     # ragged split point
        for lo, hi in ((0, k), (k, m)):
            shards.append((hi - lo, n))
            full_rows.append(m)
            parts.append((i, lo, hi))
    W = [gen_tensor(s, 0.02, seed_of(73, 0, i, "W"), "cuda") for i, s in enumerate(full)]
    G = [gen_tensor(s, 1e-3, seed_of(73, 0, i, "G"), "cuda", "bf16") for i, s in enumerate(full)]
    M = [gen_tensor(s, 1e-3, seed_of(73, 0, i, "M"), "cuda") for i, s in enumerate(full)]
    ref = [R.muon_step(W[i].double().cpu().numpy(), G[i].double().cpu().numpy(), M[i].double().cpu().numpy(),
                       LR, WD, MU, 0, "rownorm", 1e-8) for i in range(len(full))]
    Ws = [W[i][lo:hi].clone() for i, lo, hi in parts]
    Gs = [G[i][lo:hi].clone() for i, lo, hi in parts]
    Ms = [M[i][lo:hi].clone() for i, lo, hi in parts]
    plan = lib.MuonPlan(shards, "bf16", full_rows=full_rows)
    n_col = plan.info()["colsq_len"]
    offs, off = [], 0
    for (rows, n), f in zip(shards, full_rows):
        offs.append(off if f > n else None)
        off += (n + 3) // 4 * 4 if f > n else 0
    assert n_col == off
    colsq = torch.full((n_col,), float("nan"), device="cuda")
    plan.rownorm_shard_stats(Ws, Gs, Ms, LR, WD, colsq)
    for j in range(0, len(shards), 2):                 # the two blocks of one matrix
        if offs[j] is None:
            continue
        n = shards[j][1]
        a, b = colsq[offs[j]:offs[j] + n].clone(), colsq[offs[j + 1]:offs[j + 1] + n].clone()
        colsq[offs[j]:offs[j] + n] = a + b
        colsq[offs[j + 1]:offs[j + 1] + n] = a + b
    plan.rownorm_shard_apply(Ws, Gs, Ms, LR, WD, colsq)
    plan.sync()
    with pytest.raises(lib.MuonError) as ei:
        plan.step(Ws, Gs, Ms, LR, WD, MU)               # a shard plan runs RowNorm only
    assert ei.value.code == lib.MUON_ERR_UNSUPPORTED
    for i in range(len(full)):
        w = torch.cat([Ws[j] for j, (ii, _, _) in enumerate(parts) if ii == i]).double().cpu().numpy()
        m = torch.cat([Ms[j] for j, (ii, _, _) in enumerate(parts) if ii == i]).double().cpu().numpy()
        assert rel(m, ref[i][1]) <= TOL_FP32, (full[i], rel(m, ref[i][1]))
        assert rel(w, ref[i][0]) <= TOL_FP32, (full[i], rel(w, ref[i][0]))
    plan.close()


def test_select_precision_splits_only_where_the_plain_recipe_misses_the_tolerance():
    """select_precision on the caller's data: per oriented shape, the plain recipe, split
    level 1 and the reference (level 2) run on a sample; 256 x 256 (plain measured at
    2.1e-2) must take level 1, the rectangular 300 x 700 (3.5e-3) stays plain.  The chosen
    per-matrix levels then build the plan (precision_of), which meets the oracle's bar on
    every matrix, and the caller's tensors are left untouched by the selection."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(256, 256)] * 3 + [(300, 700)] * 2 + [(1024, 1024)] + [(96, 96)]
    inputs = host_inputs(shapes, "bf16", base_seed=74)
    W = [w.cuda() for w, _, _ in inputs]
    G = [g.cuda() for _, g, _ in inputs]
    M = [m.cuda() for _, _, m in inputs]
    W0, M0 = [w.clone() for w in W], [m.clone() for m in M]
    levels, report = lib.select_precision(shapes, "bf16", W, G, M, tol=1e-2, sample=2)
    for a, b in zip(W + M, W0 + M0):
        assert torch.equal(a, b)
    assert report[(256, 256)]["chosen"] == 1, report[(256, 256)]
    assert report[(300, 700)]["chosen"] == -1, report[(300, 700)]
    assert report[(256, 256)]["candidates"][-1]["err"] > 1e-2
    assert report[(256, 256)]["candidates"][1]["err"] <= 1e-2
    assert levels[:3] == [1] * 3 and levels[3:5] == [-1] * 2
    res = run_step(shapes, "bf16", inputs=inputs, precision_of=levels)
    split_shapes = {min(s) for s, lv in zip(shapes, levels) if lv > 0 and min(s) > 128}
    assert res["plan"].info()["split_buckets"] == len(split_shapes)
    for i in range(len(shapes)):
        assert_ns(res, i)


def test_measured_costs_drive_the_owner_partition():
    """measure_costs times every oriented shape on this GPU; the owner partition over those
    costs covers every matrix once and keeps the ranks' loads within the largest cost."""
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(512, 2048)] * 6 + [(2048, 512)] * 2 + [(1024, 1024)] * 3 + [(128, 1024)] * 8
    costs = lib.measure_costs(shapes, "bf16", sample=2, reps=2)
    assert len(costs) == len(shapes) and all(c > 0 for c in costs)
    assert costs[0] == costs[6]                          # one oriented shape, one cost
    owners, loads = lib.partition_owners(shapes, 3, costs)
    assert sorted(set(owners)) == [0, 1, 2]
    assert abs(sum(loads) - sum(costs)) < 1e-6 * sum(costs)
    assert max(loads) - min(loads) <= max(costs) + 1e-9


def test_plan_follows_new_tensors_between_steps():
    """One plan, three NS steps on two different sets of device tensors (A, B, A): the plan
    uploads the new pointers and re-encodes the W maps of its final products (fused r <= 128
    and batched, both orientations) whenever they change.  Every step against the oracle:
    M and W given O at 1e-5, O within the bar."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    shapes = [(128, 3584), (3584, 128), (300, 700), (700, 300), (96, 96), (256, 1024)]
    plan = lib.MuonPlan(shapes, "bf16", keep_update=True)
    sets = []
    for seed in (61, 62):
        inp = host_inputs(shapes, "bf16", seed)
        sets.append(([x[0].cuda() for x in inp], [x[1].cuda() for x in inp], [x[2].cuda() for x in inp]))
    assert all(a.data_ptr() != b.data_ptr() for a, b in zip(sets[0][0], sets[1][0]))
    for k in (0, 1, 0):
        W, G, M = sets[k]
        w0 = [w.double().cpu().numpy() for w in W]
        m0 = [m.double().cpu().numpy() for m in M]
        plan.step(W, G, M, LR, WD, MU, 5, "ns")
        plan.sync()
        for i, (m, n) in enumerate(shapes):
            g = G[i].double().cpu().numpy()
            m_ref = R.momentum(m0[i], g, MU)
            assert rel(M[i].cpu().numpy(), m_ref) <= TOL_FP32, (k, i)
            o = plan.debug_update(i).double().cpu().numpy()
            assert rel(W[i].cpu().numpy(), R.apply_update(w0[i], o, LR, WD, R.update_scale(m, n))) <= TOL_FP32, (k, i)
            e = rel(o, R.orthogonalised_update(R.nesterov(m_ref, g, MU), 5, form="gram"))
            assert e <= TOL_O, (k, i, shapes[i], e)
    plan.close()
