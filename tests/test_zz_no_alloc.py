"""The allocation-free RowNorm entry point (muon_rownorm_matrix_noalloc), called
through the C ABI: against the planned RowNorm step (muon_rownorm_step) on the
same inputs, two calls in a row, and against the fp64 oracle.  It serves callers
that may not allocate device memory (framework-owned allocators, fixed memory
budgets, loops that cannot take cudaMalloc's implicit synchronisation); its
column statistics live in a fixed scratch array inside the library."""
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
    a = np.asarray(a.double().cpu().numpy() if hasattr(a, "cpu") else a, np.float64)
    b = np.asarray(b.double().cpu().numpy() if hasattr(b, "cpu") else b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def noalloc(lib, w, g, m, gdtype, stream):
    rows, cols = w.shape
    return lib.load().muon_rownorm_matrix_noalloc(
        ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(m.data_ptr()), rows, cols,
        gdtype, LR, WD, MU, EPS, ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("shape,gdt", [((1024, 256), "bf16"), ((12288, 2048), "bf16"), ((1000, 333), "f32"),
                                       ((256, 1024), "bf16"), ((37, 4099), "f32")])
def test_noalloc_matches_planned_rownorm_twice(lib, shape, gdt):
    """Two steps in a row on a non-default stream, each against the planned step."""
    import torch
    from workloads import gen_tensor, seed_of
    gdtype = lib.MUON_BF16 if gdt == "bf16" else lib.MUON_F32
    w0 = gen_tensor(shape, 0.02, seed_of(50, 0, 0, "W"), "cuda")
    m0 = gen_tensor(shape, 1e-3, seed_of(50, 0, 0, "M"), "cuda")
    grads = [gen_tensor(shape, 1e-3, seed_of(50, t, 0, "G"), "cuda", gdt) for t in range(2)]
    plan = lib.MuonPlan([shape], gdt)
    w_ref, m_ref = w0.clone(), m0.clone()
    w_na, m_na = w0.clone(), m0.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for t in range(2):
        plan.rownorm_step([w_ref], [grads[t]], [m_ref], LR, WD, MU, EPS)
        st = noalloc(lib, w_na, grads[t], m_na, gdtype, side)
        assert st == lib.MUON_OK, lib.muon_status_string(st)
        torch.cuda.synchronize()
        assert rel(m_na, m_ref) <= TOL, (t, rel(m_na, m_ref))
        assert rel(w_na, w_ref) <= TOL, (t, rel(w_na, w_ref))
    plan.sync()
    plan.close()


@pytest.mark.parametrize("shape,gdt", [((1000, 333), "bf16"), ((333, 1000), "f32"), ((64, 64), "bf16")])
def test_noalloc_matches_the_oracle_and_writes_nothing_else(lib, shape, gdt):
    """One step per orientation against the fp64 oracle's RowNorm step (W and M at
    1e-5), with W, G and M views into larger allocations: 4096 elements of guard on
    each side stay bit-identical and G is untouched."""
    import torch
    from oracle import muon_ref as R
    from workloads import gen_tensor, seed_of
    gdtype = lib.MUON_BF16 if gdt == "bf16" else lib.MUON_F32
    w0 = gen_tensor(shape, 0.02, seed_of(51, 0, 0, "W"))
    m0 = gen_tensor(shape, 1e-3, seed_of(51, 0, 0, "M"))
    g0 = gen_tensor(shape, 1e-3, seed_of(51, 0, 0, "G"), dtype=gdt)
    guard = 4096
    views, bufs = [], []
    for t in (w0, g0, m0):
        n = t.numel()
        buf = torch.randn(n + 2 * guard, device="cuda").to(t.dtype)
        view = buf[guard:guard + n].view(t.shape)
        view.copy_(t.cuda())
        views.append(view)
        bufs.append((buf, n, buf.clone()))
    w, g, m = views
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    st = noalloc(lib, w, g, m, gdtype, side)
    assert st == lib.MUON_OK, lib.muon_status_string(st)
    torch.cuda.synchronize()
    w_ref, m_ref, _ = R.muon_step(w0.double().numpy(), g0.double().numpy(), m0.double().numpy(), LR, WD, MU, 0,
                                  "rownorm", EPS)
    assert rel(m, m_ref) <= TOL, rel(m, m_ref)
    assert rel(w, w_ref) <= TOL, rel(w, w_ref)
    for buf, n, ref in bufs:
        assert torch.equal(buf[:guard], ref[:guard]) and torch.equal(buf[guard + n:], ref[guard + n:])
    assert torch.equal(g.cpu(), g0)


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
