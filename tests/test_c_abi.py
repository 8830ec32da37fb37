"""The C ABI from C: tests/c_abi/abi_check.c is compiled as C99 with warnings as
errors against include/muon.h, linked against the built library, and run on the
CPU.  The layouts and figures it prints must match what the Python binding sees."""
import ctypes
import os
import shutil
import subprocess

import pytest

import matrix_orthogonalising_optimizer_muon_gb300 as mu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mu.load()   # builds the library if needed
    libdir = os.path.dirname(mu.LIB)
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_check")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", exe, "-L", libdir, "-lmuon_gb300",
           "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = {}
    for line in r.stdout.splitlines():
        k, _, v = line.partition(" ")
        out[k] = v
    return out


def test_c_sees_the_binding_layouts(c_output):
    for cname, cls in (("muon_plan_opts", mu.MuonPlanOpts), ("muon_plan_info_t", mu.MuonPlanInfo)):
        assert int(c_output["sizeof." + cname]) == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert int(c_output["%s.%s" % (cname, f)]) == getattr(cls, f).offset, (cname, f)
    assert int(c_output["sizeof.muon_shape"]) == ctypes.sizeof(mu.MuonShape)


def test_c_calls_match_the_binding(c_output):
    lib = mu.load()
    for code in range(mu.MUON_OK, mu.MUON_ERR_NONFINITE + 1):
        assert c_output["status.%d" % code] == lib.muon_status_string(code).decode()
    layer = [(3584, 3584), (512, 3584), (512, 3584), (3584, 3584), (18944, 3584), (18944, 3584), (3584, 18944)]
    ref = mu.plan_workspace_size(layer)
    assert int(c_output["layer.status"]) == mu.MUON_OK
    assert int(c_output["layer.bytes"]) == ref["workspace_bytes"]
    assert int(c_output["layer.buckets"]) == ref["n_buckets"] == 3
    assert int(c_output["layer.chunks"]) == 1
    ref4 = mu.plan_workspace_size(layer, chunks=4)
    assert int(c_output["chunked.status"]) == mu.MUON_OK
    assert int(c_output["chunked.bytes"]) == ref4["workspace_bytes"]
    assert int(c_output["chunked.chunks"]) == ref4["n_chunks"] >= 4
    assert int(c_output["bad.create"]) == mu.MUON_ERR_INVALID_ARG
    assert int(c_output["bad.step"]) == mu.MUON_ERR_INVALID_ARG
