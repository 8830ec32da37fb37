"""Host-side checks that need no GPU: the library builds, loads and exports every
entry point declared in include/muon.h; argument validation that happens before
any CUDA call."""
import ctypes
import os
import re

import pytest

import matrix_orthogonalising_optimizer_muon_gb300 as mu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "muon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    names = declared_functions()
    assert "muon_step" in names and "muon_plan_create" in names and "muon_rownorm_step" in names
    assert sorted(mu.EXPORTED) == names


def struct_fields(name):
    """(field, bytes) of a typedef struct in include/muon.h, in order."""
    src = open(os.path.join(ROOT, "include", "muon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\}\s*" + name + r"\s*;", src).group(1)
    size = {"int32_t": 4, "int64_t": 8}
    out = []
    for t, ptr, f in re.findall(r"\b(int32_t|int64_t)\s*(\*?)\s*(\w+)\s*;", body):
        out.append((f, 8 if ptr else size[t]))   # pointers are 8 bytes on both hosts
    return out


def test_struct_layouts_match_the_header():
    for name, cls in (("muon_plan_opts", mu.MuonPlanOpts), ("muon_plan_info_t", mu.MuonPlanInfo)):
        fields = struct_fields(name)
        assert [f for f, _ in fields] == [f for f, _ in cls._fields_], name
        assert [b for _, b in fields] == [ctypes.sizeof(t) for _, t in cls._fields_], name
        assert ctypes.sizeof(cls) == sum(b for _, b in fields), name


def test_library_exports_every_declared_symbol():
    lib = mu.load()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    lib = mu.load()
    for code in range(7):
        s = lib.muon_status_string(code).decode()
        assert s.startswith("MUON_")
    assert b"UNKNOWN" in lib.muon_status_string(99)


def test_plan_create_rejects_bad_arguments_before_cuda():
    lib = mu.load()
    h = ctypes.c_void_p()
    shapes = (mu.MuonShape * 2)(mu.MuonShape(4, 8), mu.MuonShape(0, 3))
    assert lib.muon_plan_create(shapes, 2, mu.MUON_BF16, None, ctypes.byref(h)) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_create(shapes, 0, mu.MUON_BF16, None, ctypes.byref(h)) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_create(shapes, 1, 7, None, ctypes.byref(h)) == mu.MUON_ERR_UNSUPPORTED
    assert lib.muon_plan_create(None, 1, mu.MUON_BF16, None, ctypes.byref(h)) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_step(None, None, None, None, 0.1, 0.1, 0.9, 5, 0, None) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_sync(None, None) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_plan_tune(None, None, None, None, 0.1, 0.1, 0.9, 3, None, None) == mu.MUON_ERR_INVALID_ARG
    assert lib.muon_step_host(None, None, None, None, None, None, 0.1, 0.1, 0.9, 5, 0, None) == \
        mu.MUON_ERR_INVALID_ARG
    one = (mu.MuonShape * 1)(mu.MuonShape(4, 8))
    for bad in (mu.MuonPlanOpts(chunks=-1), mu.MuonPlanOpts(workspace_bytes=-1)):
        assert lib.muon_plan_create(one, 1, mu.MUON_BF16, ctypes.byref(bad), ctypes.byref(h)) == \
            mu.MUON_ERR_INVALID_ARG
    big = (mu.MuonShape * 1)(mu.MuonShape(1 << 21, 4))
    assert lib.muon_plan_create(big, 1, mu.MUON_F32, None, ctypes.byref(h)) == mu.MUON_ERR_UNSUPPORTED


def test_schedule_helper():
    class FakePlan:
        def __init__(self):
            self.calls = []

        def step(self, *a, **k):
            self.calls.append("ns")

        def rownorm_step(self, *a, **k):
            self.calls.append("rownorm")

    p = FakePlan()
    sched = mu.PeriodicRowNormMuon(p, k=4)
    modes = [sched.step([], [], [], 0.02, 0.1) for _ in range(8)]
    assert modes == ["ns", "rownorm", "rownorm", "rownorm"] * 2
    assert p.calls == modes
    with pytest.raises(ValueError):
        mu.PeriodicRowNormMuon(p, k=0)


def test_schedule_resumes_from_its_state():
    class FakePlan:
        def __init__(self):
            self.calls = []

        def step(self, *a, **k):
            self.calls.append("ns")

        def rownorm_step(self, *a, **k):
            self.calls.append("rownorm")

    whole = mu.PeriodicRowNormMuon(FakePlan(), k=4, eps=1e-7)
    ref = [whole.step([], [], [], 0.02, 0.1) for _ in range(11)]
    first = mu.PeriodicRowNormMuon(FakePlan(), k=4, eps=1e-7)
    got = [first.step([], [], [], 0.02, 0.1) for _ in range(6)]
    state = dict(first.state_dict())
    resumed = mu.PeriodicRowNormMuon(FakePlan(), k=9)   # settings come from the state
    resumed.load_state_dict(state)
    assert (resumed.k, resumed.eps, resumed.t) == (4, 1e-7, 6)
    got += [resumed.step([], [], [], 0.02, 0.1) for _ in range(5)]
    assert got == ref
    for bad in ({"t": -1, "k": 4}, {"t": 0, "k": 0}):
        with pytest.raises(ValueError):
            resumed.load_state_dict(bad)
