"""The allocation-free RowNorm entry point (muon_rownorm_matrix_noalloc), called
through the C ABI, against the planned RowNorm step (muon_rownorm_step) on the
same inputs, two calls in a row.  It serves callers that may not allocate
device memory (framework-owned allocators, fixed memory budgets, loops that
cannot take cudaMalloc's implicit synchronisation); its column statistics
live in a fixed scratch array inside the library."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL = 1e-5
LR, WD, MU, EPS = 0.02, 0.1, 0.95, 1e-8


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import matrix_orthogonalising_optimizer_muon_gb300 as mu
    return mu


def rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("shape,gdt", [((1024, 256), "bf16"), ((12288, 2048), "bf16"), ((1000, 333), "f32"),
                                       ((256, 1024), "bf16"), ((37, 4099), "f32")])
def test_noalloc_matches_planned_rownorm_twice(lib, shape, gdt):
    import torch
    from workloads import gen_tensor, seed_of
    m, n = shape
    gdtype = lib.MUON_BF16 if gdt == "bf16" else lib.MUON_F32
    w0 = gen_tensor(shape, 0.02, seed_of(50, 0, 0, "W"), "cuda")
    m0 = gen_tensor(shape, 1e-3, seed_of(50, 0, 0, "M"), "cuda")
    grads = [gen_tensor(shape, 1e-3, seed_of(50, t, 0, "G"), "cuda", gdt) for t in range(2)]
    # planned path
    plan = lib.MuonPlan([shape], gdt)
    w_ref, m_ref = w0.clone(), m0.clone()
    # allocation-free path
    w_na, m_na = w0.clone(), m0.clone()
    stream = torch.cuda.current_stream()
    h = ctypes.c_void_p(stream.cuda_stream)
    for t in range(2):
        plan.rownorm_step([w_ref], [grads[t]], [m_ref], LR, WD, MU, EPS)
        st = lib.load().muon_rownorm_matrix_noalloc(
            ctypes.c_void_p(w_na.data_ptr()), ctypes.c_void_p(grads[t].data_ptr()),
            ctypes.c_void_p(m_na.data_ptr()), m, n, gdtype, LR, WD, MU, EPS, h)
        assert st == lib.MUON_OK, lib.muon_status_string(st)
        torch.cuda.synchronize()
        assert rel(m_na, m_ref) <= TOL, (t, rel(m_na, m_ref))
        assert rel(w_na, w_ref) <= TOL, (t, rel(w_na, w_ref))
    plan.sync()
    plan.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    import torch
    w = torch.zeros(4, device="cuda")
    g = torch.zeros(4, device="cuda")
    mo = torch.zeros(4, device="cuda")
    f = lib.load().muon_rownorm_matrix_noalloc
    args = [ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(mo.data_ptr())]
    # ceil(70000 / 64) * 1000 + 1000 floats > 2^20: refused before any launch
    st = f(*args, 70000, 1000, lib.MUON_F32, LR, WD, MU, EPS, None)
    assert st == lib.MUON_ERR_UNSUPPORTED
    assert f(*args, 4, 0, lib.MUON_F32, LR, WD, MU, EPS, None) == lib.MUON_ERR_INVALID_ARG
    assert f(*args, 2, 2, lib.MUON_F32, LR, WD, 1.0, EPS, None) == lib.MUON_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert float(w.abs().sum()) == 0.0 and float(mo.abs().sum()) == 0.0
