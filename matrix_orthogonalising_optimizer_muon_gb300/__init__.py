"""Python binding of libmuon_gb300.so, a single-GPU Muon optimizer step for GB300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides the device memory and the stream.  There is no
fallback: if the library cannot be loaded, every entry point raises.

The C entry points keep their names (``muon_plan_create``, ``muon_step``,
``muon_rownorm_step``, ``muon_sync``, ``muon_debug_copy_update``,
``muon_debug_copy_workspace``, ``muon_plan_info``, ``muon_stage_times``,
``muon_status_string``, ``muon_plan_destroy`` and the rest of the header);
``MuonPlan`` wraps them for torch tensors, ``plan_workspace_size`` sizes a plan on
the host alone (``muon_plan_workspace_size``), and ``PeriodicRowNormMuon`` adds the step schedule of periodic
RowNorm Muon (full NS5 every K steps, RowNorm otherwise; "Scaling Muon for
Diffusion Transformers", sec. 3).  ``DistributedMuon`` runs the step across the
ranks of a torch.distributed group with one owner per matrix (``partition_owners``,
the library's ``muon_partition``) and broadcasts the updated parameters.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB, build, up_to_date

__all__ = [
    "MuonError", "MuonPlan", "PeriodicRowNormMuon", "DistributedMuon", "ShardedRowNorm", "partition_owners",
    "select_precision", "measure_costs",
    "plan_workspace_size", "load", "build",
    "MUON_OK", "MUON_ERR_INVALID_ARG", "MUON_ERR_UNSUPPORTED", "MUON_ERR_OOM",
    "MUON_ERR_CUDA", "MUON_ERR_TIMEOUT", "MUON_ERR_NONFINITE", "MUON_F32", "MUON_BF16",
    "MUON_MODE_NS", "MUON_MODE_ROWNORM", "EXPORTED",
]

MUON_OK, MUON_ERR_INVALID_ARG, MUON_ERR_UNSUPPORTED, MUON_ERR_OOM = 0, 1, 2, 3
MUON_ERR_CUDA, MUON_ERR_TIMEOUT, MUON_ERR_NONFINITE = 4, 5, 6
MUON_F32, MUON_BF16 = 0, 1
MUON_MODE_NS, MUON_MODE_ROWNORM = 0, 1

# Newton-Schulz steps and momentum the pages use ("Muon is Scalable" blog).
DEFAULT_NS_STEPS = 5
DEFAULT_MU = 0.95


class MuonShape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class MuonPlanOpts(ctypes.Structure):
    _fields_ = [("keep_update", ctypes.c_int32), ("timing", ctypes.c_int32),
                ("single_sm_gemm", ctypes.c_int32), ("generic_small", ctypes.c_int32),
                ("chain_clusters", ctypes.c_int32), ("max_ns_steps", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("chunks", ctypes.c_int32),
                ("full_symmetric", ctypes.c_int32), ("small_fp32", ctypes.c_int32),
                ("check_finite", ctypes.c_int32), ("precision", ctypes.c_int32), ("split_max_r", ctypes.c_int32),
                ("full_rows", ctypes.POINTER(ctypes.c_int64)), ("precision_of", ctypes.POINTER(ctypes.c_int32))]


class MuonPlanInfo(ctypes.Structure):
    _fields_ = [("n_matrices", ctypes.c_int32), ("n_buckets", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("launches_last_step", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("n_chunks", ctypes.c_int32), ("lower_chunks", ctypes.c_int32),
                ("tuned_candidates", ctypes.c_int32), ("chain_clusters", ctypes.c_int32),
                ("split_buckets", ctypes.c_int32), ("fp32_buckets", ctypes.c_int32), ("colsq_len", ctypes.c_int64)]


_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
# name -> (restype, argtypes); every function declared in include/muon.h
EXPORTED = {
    "muon_plan_create": (ctypes.c_int, [ctypes.POINTER(MuonShape), ctypes.c_int32, ctypes.c_int,
                                        ctypes.POINTER(MuonPlanOpts), ctypes.POINTER(_P)]),
    "muon_plan_destroy": (None, [_P]),
    "muon_plan_workspace_size": (ctypes.c_int, [ctypes.POINTER(MuonShape), ctypes.c_int32, ctypes.c_int,
                                                ctypes.POINTER(MuonPlanOpts), ctypes.POINTER(ctypes.c_int64),
                                                ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "muon_debug_wait_timeout": (ctypes.c_int, [_P, ctypes.c_int32, _P]),
    "muon_step": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                 ctypes.c_int32, ctypes.c_int, _P]),
    "muon_step_ex": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_int32, ctypes.POINTER(ctypes.c_float), ctypes.c_int32, _P]),
    "muon_step_host": (ctypes.c_int, [_P, _PP, _PP, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_float, ctypes.c_int32, ctypes.c_int, _P]),
    "muon_rownorm_step": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float,
                                         ctypes.c_float, ctypes.c_float, _P]),
    "muon_sync": (ctypes.c_int, [_P, _P]),
    "muon_plan_tune": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int32, ctypes.POINTER(ctypes.c_float), _P]),
    "muon_debug_copy_update": (ctypes.c_int, [_P, ctypes.c_int32, _P, _P]),
    "muon_debug_update_error": (ctypes.c_int, [_P, ctypes.c_int32, _P, ctypes.POINTER(ctypes.c_double), _P]),
    "muon_debug_copy_workspace": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, _P,
                                                 ctypes.POINTER(ctypes.c_int32), _P]),
    "muon_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "muon_last_error_detail": (ctypes.c_char_p, []),
    "muon_plan_info": (ctypes.c_int, [_P, ctypes.POINTER(MuonPlanInfo)]),
    "muon_stage_times": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_float),
                                        ctypes.POINTER(ctypes.c_double), ctypes.c_int32]),
    "muon_rownorm_shard_stats": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                ctypes.c_float, _P, _P]),
    "muon_rownorm_shard_apply": (ctypes.c_int, [_P, _PP, _PP, _PP, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                ctypes.c_float, _P, _P]),
    "muon_partition": (ctypes.c_int, [ctypes.POINTER(MuonShape), ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_double)]),
    "muon_rownorm_matrix_noalloc": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                   ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_float, _P]),
}

_lib = None


def load(path: str | None = None):
    """Load (building first if missing) the CUDA library and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        path = LIB
        if not up_to_date():
            build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTED.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB:
        _lib = lib
    return lib


class MuonError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        lib = load()
        msg = lib.muon_status_string(code).decode()
        if code == MUON_ERR_CUDA:
            msg += " (%s)" % lib.muon_last_error_detail().decode()
        super().__init__("%s: %s" % (where, msg))


def _check(code: int, where: str):
    if code != MUON_OK:
        raise MuonError(code, where)


def muon_status_string(code: int) -> str:
    return load().muon_status_string(code).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr_array(ptrs):
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def _plan_args(shapes, grad_dtype, keep_update=False, timing=False, single_sm_gemm=False,
               generic_small=False, chain_clusters=0, workspace_bytes=0, max_ns_steps=0, chunks=0,
               full_symmetric=False, small_fp32=0, check_finite=False, precision=0, split_max_r=0,
               full_rows=None, precision_of=None):
    """(shape list, MuonShape array, dtype code, MuonPlanOpts) of a plan's arguments.  The
    options keep a reference to the full_rows array (read by the library during creation)."""
    shapes = [(int(m), int(n)) for m, n in shapes]
    arr = (MuonShape * len(shapes))(*[MuonShape(m, n) for m, n in shapes])
    fr = None
    if full_rows is not None:
        if len(full_rows) != len(shapes):
            raise ValueError("full_rows needs one entry per matrix")
        fr = (ctypes.c_int64 * len(shapes))(*[int(x) for x in full_rows])
    po = None
    if precision_of is not None:
        if len(precision_of) != len(shapes):
            raise ValueError("precision_of needs one entry per matrix")
        po = (ctypes.c_int32 * len(shapes))(*[int(x) for x in precision_of])
    opts = MuonPlanOpts(1 if keep_update else 0, 1 if timing else 0, 1 if single_sm_gemm else 0,
                        1 if generic_small else 0, int(chain_clusters), int(max_ns_steps),
                        int(workspace_bytes), int(chunks), 1 if full_symmetric else 0, int(small_fp32),
                        1 if check_finite else 0, int(precision), int(split_max_r),
                        ctypes.cast(fr, ctypes.POINTER(ctypes.c_int64)) if fr is not None else None,
                        ctypes.cast(po, ctypes.POINTER(ctypes.c_int32)) if po is not None else None)
    opts._arrays = (fr, po)
    return shapes, arr, {"bf16": MUON_BF16, "f32": MUON_F32}[grad_dtype], opts


def plan_workspace_size(shapes, grad_dtype: str = "bf16", **opts) -> dict:
    """What ``MuonPlan(shapes, grad_dtype, **opts)`` would build, computed on the host alone
    (``muon_plan_workspace_size``; no GPU needed): the device workspace bytes it would
    allocate, its (r, c) buckets and its chunks."""
    lib = load()
    shapes, arr, gd, o = _plan_args(shapes, grad_dtype, **opts)
    nbytes, nb, nc = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib.muon_plan_workspace_size(arr, len(shapes), gd, ctypes.byref(o), ctypes.byref(nbytes),
                                        ctypes.byref(nb), ctypes.byref(nc)), "muon_plan_workspace_size")
    return {"workspace_bytes": nbytes.value, "n_buckets": nb.value, "n_chunks": nc.value}


class MuonPlan:
    """A planned Muon step over a fixed list of matrix shapes (``muon_plan_create``).

    ``step`` takes lists of torch tensors: params (fp32), grads (``grad_dtype``)
    and momentum (fp32), all contiguous CUDA tensors of the planned shapes, and
    updates params and momentum in place on the current stream."""

    def __init__(self, shapes, grad_dtype: str = "bf16", keep_update: bool = False,
                 timing: bool = False, single_sm_gemm: bool = False, generic_small: bool = False,
                 chain_clusters: int = 0, workspace_bytes: int = 0, max_ns_steps: int = 0, chunks: int = 0,
                 full_symmetric: bool = False, small_fp32: int = 0, check_finite: bool = False,
                 precision: int = 0, split_max_r: int = 0, full_rows=None, precision_of=None):
        self.lib = load()
        self.shapes, arr, gd, opts = _plan_args(shapes, grad_dtype, keep_update, timing, single_sm_gemm,
                                                generic_small, chain_clusters, workspace_bytes, max_ns_steps,
                                                chunks, full_symmetric, small_fp32, check_finite, precision,
                                                split_max_r, full_rows, precision_of)
        self.grad_dtype = grad_dtype
        h = ctypes.c_void_p()
        _check(self.lib.muon_plan_create(arr, len(self.shapes), gd, ctypes.byref(opts),
                                         ctypes.byref(h)), "muon_plan_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.muon_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---------------------------------------------------------------- marshalling
    def _pointers(self, params, grads, momentum):
        import torch
        n = len(self.shapes)
        if not (len(params) == len(grads) == len(momentum) == n):
            raise ValueError("expected %d params, grads and momentum tensors" % n)
        gdt = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        for i, (w, g, m) in enumerate(zip(params, grads, momentum)):
            shp = self.shapes[i]
            for t, dt, name in ((w, torch.float32, "param"), (g, gdt, "grad"),
                                (m, torch.float32, "momentum")):
                if tuple(t.shape) != shp or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
                    raise ValueError("%s %d: need a contiguous CUDA %s tensor of shape %s, got %s %s"
                                     % (name, i, dt, shp, t.dtype, tuple(t.shape)))
        return (_ptr_array([t.data_ptr() for t in params]),
                _ptr_array([t.data_ptr() for t in grads]),
                _ptr_array([t.data_ptr() for t in momentum]))

    def step(self, params, grads, momentum, lr: float, wd: float, mu: float = DEFAULT_MU,
             ns_steps: int = DEFAULT_NS_STEPS, mode: str = "ns", stream=None, coeffs=None, restart: int = 0):
        """One Muon step (``muon_step``; ``muon_step_ex`` when NS coefficients (a, b, c)
        or a restart period are given)."""
        w, g, m = self._pointers(params, grads, momentum)
        self._step(w, g, m, lr, wd, mu, ns_steps, mode, 1e-8, stream, coeffs, restart)

    def _step(self, w, g, m, lr, wd, mu, ns_steps, mode, eps, stream, coeffs, restart):
        if mode == "rownorm":
            _check(self.lib.muon_rownorm_step(self.handle, w, g, m, lr, wd, mu, eps,
                                              _stream_handle(stream)), "muon_rownorm_step")
        elif mode != "ns":
            raise ValueError("mode must be 'ns' or 'rownorm'")
        elif coeffs is None and not restart:
            _check(self.lib.muon_step(self.handle, w, g, m, lr, wd, mu, ns_steps, MUON_MODE_NS,
                                      _stream_handle(stream)), "muon_step")
        else:
            abc = None if coeffs is None else (ctypes.c_float * 3)(*[float(x) for x in coeffs])
            _check(self.lib.muon_step_ex(self.handle, w, g, m, lr, wd, mu, ns_steps, abc, int(restart),
                                         _stream_handle(stream)), "muon_step_ex")

    def step_host(self, params, grads, momentum, grads_host, params_host, lr: float, wd: float,
                  mu: float = DEFAULT_MU, ns_steps: int = DEFAULT_NS_STEPS, mode: str = "ns", stream=None):
        """``muon_step_host``: gradients copied in from the CPU tensors ``grads_host`` (into the
        CUDA tensors ``grads``), the updated params copied back into the CPU tensors
        ``params_host`` (or not, if None), overlapped with the compute chunk by chunk.  Pinned
        CPU tensors keep the copies asynchronous; synchronise the stream before reading
        ``params_host``."""
        import torch
        w, g, m = self._pointers(params, grads, momentum)
        n = len(self.shapes)
        gdt = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        outs = [] if params_host is None else list(params_host)
        if len(grads_host) != n or (params_host is not None and len(outs) != n):
            raise ValueError("expected %d host tensors" % n)
        for i in range(n):
            pairs = [(grads_host[i], gdt, "host grad")] + ([(outs[i], torch.float32, "host param")] if outs else [])
            for t, dt, name in pairs:
                if tuple(t.shape) != self.shapes[i] or t.dtype != dt or t.is_cuda or not t.is_contiguous():
                    raise ValueError("%s %d: need a contiguous CPU %s tensor of shape %s" % (name, i, dt,
                                                                                            self.shapes[i]))
        gh = _ptr_array([t.data_ptr() for t in grads_host])
        wh = _ptr_array([t.data_ptr() for t in outs]) if outs else None
        md = {"ns": MUON_MODE_NS, "rownorm": MUON_MODE_ROWNORM}.get(mode)
        if md is None:
            raise ValueError("mode must be 'ns' or 'rownorm'")
        _check(self.lib.muon_step_host(self.handle, w, g, m, gh, wh, lr, wd, mu, ns_steps, md,
                                       _stream_handle(stream)), "muon_step_host")

    def rownorm_step(self, params, grads, momentum, lr: float, wd: float, mu: float = DEFAULT_MU,
                     eps: float = 1e-8, stream=None):
        """One RowNorm step (``muon_rownorm_step``)."""
        w, g, m = self._pointers(params, grads, momentum)
        _check(self.lib.muon_rownorm_step(self.handle, w, g, m, lr, wd, mu, eps,
                                          _stream_handle(stream)), "muon_rownorm_step")

    def rownorm_shard_stats(self, params, grads, momentum, lr: float, wd: float, colsq, mu: float = DEFAULT_MU,
                            eps: float = 1e-8, stream=None):
        """``muon_rownorm_shard_stats`` on a plan created with ``full_rows``: colsq (a CUDA fp32
        tensor of ``info()['colsq_len']`` elements) receives this shard's column sums of U^2."""
        w, g, m = self._pointers(params, grads, momentum)
        _check(self.lib.muon_rownorm_shard_stats(self.handle, w, g, m, lr, wd, mu, eps,
                                                 ctypes.c_void_p(colsq.data_ptr()), _stream_handle(stream)),
               "muon_rownorm_shard_stats")

    def rownorm_shard_apply(self, params, grads, momentum, lr: float, wd: float, colsq, mu: float = DEFAULT_MU,
                            eps: float = 1e-8, stream=None):
        """``muon_rownorm_shard_apply``: the update of the spanning matrices from colsq summed
        over every shard."""
        w, g, m = self._pointers(params, grads, momentum)
        _check(self.lib.muon_rownorm_shard_apply(self.handle, w, g, m, lr, wd, mu, eps,
                                                 ctypes.c_void_p(colsq.data_ptr()), _stream_handle(stream)),
               "muon_rownorm_shard_apply")

    def bind(self, params, grads, momentum):
        """Validate the tensors once and keep their pointer arrays for ``step_bound``.
        The tensors must stay alive and in place while bound."""
        self._bound = self._pointers(params, grads, momentum)
        self._bound_refs = (list(params), list(grads), list(momentum))

    def step_bound(self, lr: float, wd: float, mu: float = DEFAULT_MU, ns_steps: int = DEFAULT_NS_STEPS,
                   mode: str = "ns", eps: float = 1e-8, stream=None, coeffs=None, restart: int = 0):
        """``muon_step`` / ``muon_step_ex`` / ``muon_rownorm_step`` on the tensors given to ``bind``."""
        w, g, m = self._bound
        self._step(w, g, m, lr, wd, mu, ns_steps, mode, eps, stream, coeffs, restart)

    def tune(self, params, grads, momentum, lr: float, wd: float, mu: float = DEFAULT_MU, reps: int = 3,
             stream=None) -> float:
        """``muon_plan_tune``: time the plan's speed-only launch choices on these tensors (each
        candidate runs 1 + reps NS steps on them) and keep the fastest; returns its ms per step."""
        w, g, m = self._pointers(params, grads, momentum)
        ms = ctypes.c_float()
        _check(self.lib.muon_plan_tune(self.handle, w, g, m, lr, wd, mu, int(reps), ctypes.byref(ms),
                                       _stream_handle(stream)), "muon_plan_tune")
        return ms.value

    def sync(self, stream=None):
        _check(self.lib.muon_sync(self.handle, _stream_handle(stream)), "muon_sync")

    def debug_wait_timeout(self, limit_us: int, stream=None):
        """Enqueue one bounded device wait that nothing completes (``muon_debug_wait_timeout``);
        the next ``sync`` raises MuonError with MUON_ERR_TIMEOUT."""
        _check(self.lib.muon_debug_wait_timeout(self.handle, int(limit_us), _stream_handle(stream)),
               "muon_debug_wait_timeout")

    def debug_update(self, i: int, stream=None):
        """O of matrix i from the last NS step (needs keep_update), as a CUDA fp32 tensor."""
        import torch
        m, n = self.shapes[i]
        out = torch.empty((m, n), dtype=torch.float32, device="cuda")
        _check(self.lib.muon_debug_copy_update(self.handle, i, ctypes.c_void_p(out.data_ptr()),
                                               _stream_handle(stream)), "muon_debug_copy_update")
        return out

    def debug_update_error(self, i: int, ref, stream=None) -> float:
        """||O_i - ref|| / ||ref|| on the device (``muon_debug_update_error``; needs keep_update)."""
        out = ctypes.c_double()
        _check(self.lib.muon_debug_update_error(self.handle, i, ctypes.c_void_p(ref.data_ptr()), ctypes.byref(out),
                                                _stream_handle(stream)), "muon_debug_update_error")
        return out.value

    def debug_workspace(self, i: int, which: int, stream=None):
        """A workspace buffer of matrix i (``muon_debug_copy_workspace``) as a CPU fp32
        tensor of r rows (widened exactly from bf16 / fp16).  G buffers hold s*G."""
        import torch
        m, n = self.shapes[i]
        r, c = min(m, n), max(m, n)
        ld = ctypes.c_int32()
        if which == 8:
            out = torch.empty(1, dtype=torch.float32)
        else:
            width = ((c if which == 0 else r) + 7) // 8 * 8
            dt = torch.bfloat16 if which in (0, 7) else torch.float16
            out = torch.empty((r, width), dtype=dt)
        _check(self.lib.muon_debug_copy_workspace(self.handle, i, which, ctypes.c_void_p(out.data_ptr()),
                                                  ctypes.byref(ld), _stream_handle(stream)),
               "muon_debug_copy_workspace")
        if which == 8:
            return out
        assert ld.value == out.shape[1]
        return out[:, :(c if which == 0 else r)].float()

    @staticmethod
    def gram_scale(r: int) -> float:
        """The power of two s the library carries G as (s*G) in its fp16 r x r buffers."""
        import math
        return 2.0 ** round(math.log2(r))

    def info(self) -> dict:
        inf = MuonPlanInfo()
        _check(self.lib.muon_plan_info(self.handle, ctypes.byref(inf)), "muon_plan_info")
        return {k: getattr(inf, k) for k, _ in MuonPlanInfo._fields_}

    def stage_times(self):
        """Summed over the timed steps since the previous call: (ms per stage [momentum,
        syrk, rxr NS, final+apply, rownorm, fused r <= 128 step], algorithmic tensor
        flops [syrk, rxr, final] of the non-fused matrices)."""
        ms = (ctypes.c_float * 6)()
        fl = (ctypes.c_double * 3)()
        _check(self.lib.muon_stage_times(self.handle, ms, fl, 6), "muon_stage_times")
        return list(ms), list(fl)


class PeriodicRowNormMuon:
    """Periodic RowNorm Muon over one plan: step t runs NS (``ns_steps``) iff t % K == 0,
    RowNorm otherwise ("Scaling Muon for Diffusion Transformers", sec. 3; steps from 0)."""

    def __init__(self, plan: MuonPlan, k: int, eps: float = 1e-8, ns_steps: int = DEFAULT_NS_STEPS):
        if k <= 0:
            raise ValueError("K must be positive")
        self.plan, self.k, self.eps, self.ns_steps = plan, k, eps, ns_steps
        self.t = 0

    def mode_at(self, t: int) -> str:
        return "ns" if t % self.k == 0 else "rownorm"

    def step(self, params, grads, momentum, lr, wd, mu=DEFAULT_MU, stream=None) -> str:
        mode = self.mode_at(self.t)
        if mode == "ns":
            self.plan.step(params, grads, momentum, lr, wd, mu, self.ns_steps, "ns", stream)
        else:
            self.plan.rownorm_step(params, grads, momentum, lr, wd, mu, self.eps, stream)
        self.t += 1
        return mode

    def state_dict(self) -> dict:
        """The schedule's state for a checkpoint: the next step's index and its settings.
        (Momentum buffers belong to the caller and are checkpointed with the model.)"""
        return {"t": self.t, "k": self.k, "eps": self.eps, "ns_steps": self.ns_steps}

    def load_state_dict(self, state: dict) -> None:
        """Resume from ``state_dict()``: the next step runs as step ``t`` of the saved run."""
        t, k = int(state["t"]), int(state["k"])
        if t < 0 or k <= 0:
            raise ValueError("bad schedule state: t = %d, K = %d" % (t, k))
        self.t, self.k = t, k
        self.eps = float(state.get("eps", self.eps))
        self.ns_steps = int(state.get("ns_steps", self.ns_steps))


def partition_owners(shapes, world: int, costs=None):
    """Owner rank of every matrix for ``world`` GPUs (``muon_partition``: longest
    processing time first over per-matrix costs, DMuon's greedy owner assignment).
    Returns (owners, loads)."""
    lib = load()
    shapes = [(int(m), int(n)) for m, n in shapes]
    n = len(shapes)
    arr = (MuonShape * n)(*[MuonShape(m, k) for m, k in shapes])
    c = None if costs is None else (ctypes.c_double * n)(*[float(x) for x in costs])
    owner = (ctypes.c_int32 * n)()
    loads = (ctypes.c_double * int(world))()
    _check(lib.muon_partition(arr, n, int(world), c, owner, loads), "muon_partition")
    return list(owner), list(loads)


class DistributedMuon:
    """Owner-partitioned Muon step over the ranks of a torch.distributed group
    (DMuon technical summary sec. 2: each matrix has one owner rank, which keeps
    its momentum and runs its Newton-Schulz step exactly once; the updated
    parameters are then published to every other rank).

    Every rank holds every parameter matrix.  Gradients are the already reduced
    full gradients; a rank reads only the gradients and momentum of the matrices
    it owns (``owned``), so the other entries of ``grads`` and ``momentum`` may be
    None.  After its local step each owner broadcasts its updated fp32
    parameters (one NCCL broadcast per owner, from a flat buffer): the one data
    exchange of the step.  Parameters allocated by ``allocate_params`` are views
    into those flat buffers and are broadcast in place; other tensors go through
    a staging buffer (one copy on each side).  With one rank this is a plain
    ``MuonPlan`` step."""

    def __init__(self, shapes, grad_dtype: str = "bf16", group=None, costs=None, **plan_opts):
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            self.rank, self.world = dist.get_rank(group), dist.get_world_size(group)
        else:
            self.rank, self.world = 0, 1
        self.group = group
        self.grad_dtype = grad_dtype
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        self.owner, self.loads = partition_owners(self.shapes, self.world, costs)
        self.owned_by = [[i for i, o in enumerate(self.owner) if o == r] for r in range(self.world)]
        self.owned = self.owned_by[self.rank]
        self.plan = self._make_plan(plan_opts) if self.owned else None
        self._flat = None        # per owner: flat fp32 buffer of its parameters (allocate_params)
        self._views = None
        self._staging = None

    def _make_plan(self, plan_opts):
        return MuonPlan([self.shapes[i] for i in self.owned], self.grad_dtype, **plan_opts)

    def _local_step(self, params, grads, momentum, lr, wd, mu, ns_steps, mode, eps, stream):
        if mode == "ns":
            self.plan.step(params, grads, momentum, lr, wd, mu, ns_steps, "ns", stream)
        else:
            self.plan.rownorm_step(params, grads, momentum, lr, wd, mu, eps, stream)

    def allocate_params(self, device=None):
        """Parameter tensors (fp32, every matrix) laid out as one flat buffer per owner,
        so the exchange broadcasts each owner's parameters in place."""
        import torch
        self._flat, self._views = [], [None] * len(self.shapes)
        for r in range(self.world):
            idx = self.owned_by[r]
            buf = torch.empty(sum(self.shapes[i][0] * self.shapes[i][1] for i in idx), dtype=torch.float32,
                              device=device)
            off = 0
            for i in idx:
                m, n = self.shapes[i]
                self._views[i] = buf[off:off + m * n].view(m, n)
                off += m * n
            self._flat.append(buf)
        return list(self._views)

    def step(self, params, grads, momentum, lr: float, wd: float, mu: float = DEFAULT_MU,
             ns_steps: int = DEFAULT_NS_STEPS, mode: str = "ns", eps: float = 1e-8, stream=None):
        """The owned matrices' Muon step (NS or RowNorm), then the parameter exchange."""
        if mode not in ("ns", "rownorm"):
            raise ValueError("mode must be 'ns' or 'rownorm'")
        if len(params) != len(self.shapes):
            raise ValueError("expected %d parameter tensors" % len(self.shapes))
        own = self.owned
        if own:
            self._local_step([params[i] for i in own], [grads[i] for i in own], [momentum[i] for i in own],
                             lr, wd, mu, ns_steps, mode, eps, stream)
        self.exchange(params)

    def exchange(self, params):
        """Every owner broadcasts its matrices' parameters to the other ranks."""
        if self.world == 1:
            return
        import torch
        import torch.distributed as dist
        in_place = self._views is not None and all(
            p.data_ptr() == v.data_ptr() and p.shape == v.shape for p, v in zip(params, self._views))
        for r in range(self.world):
            idx = self.owned_by[r]
            if not idx:
                continue
            if in_place:
                dist.broadcast(self._flat[r], src=r, group=self.group)
                continue
            numel = sum(params[i].numel() for i in idx)
            dev = params[idx[0]].device
            if self._staging is None or self._staging.numel() < numel or self._staging.device != dev:
                self._staging = torch.empty(max(numel, max(
                    sum(self.shapes[i][0] * self.shapes[i][1] for i in ix) for ix in self.owned_by)),
                    dtype=torch.float32, device=dev)
            buf = self._staging[:numel]
            if r == self.rank:
                torch.cat([params[i].reshape(-1) for i in idx], out=buf)
            dist.broadcast(buf, src=r, group=self.group)
            if r != self.rank:
                off = 0
                for i in idx:
                    k = params[i].numel()
                    params[i].view(-1).copy_(buf[off:off + k])
                    off += k

    def sync(self, stream=None):
        if self.plan is not None:
            self.plan.sync(stream)

    def close(self):
        if self.plan is not None:
            self.plan.close()
            self.plan = None


class ShardedRowNorm:
    """RowNorm steps over dim-0 shards across the ranks of a torch.distributed group
    ("Scaling Muon for Diffusion Transformers" sec. 1 and 2.3: on RowNorm steps each rank
    keeps its block of rows of every W, G and M; only the squared norms of the RowNorm
    rows that span ranks are all-reduced).

    ``shard_shapes[i]`` is this rank's block of rows of matrix i, whose full shape is
    ``(full_rows[i], shard_shapes[i][1])``.  Matrices with full_rows <= cols have their
    RowNorm rows complete in each shard; the others (the stored columns are the RowNorm
    rows) need one sum of their per-column U^2 across ranks: one all-reduce of a single
    fp32 buffer per step, between the library's two shard calls."""

    def __init__(self, shard_shapes, full_rows, grad_dtype: str = "bf16", group=None, **plan_opts):
        import torch
        self.group = group
        self.plan = self._make_plan(shard_shapes, full_rows, grad_dtype, plan_opts)
        n = self._colsq_len()
        self.colsq = torch.zeros(max(n, 1), dtype=torch.float32, device=self._device())

    def _make_plan(self, shard_shapes, full_rows, grad_dtype, plan_opts):
        return MuonPlan(shard_shapes, grad_dtype, full_rows=full_rows, **plan_opts)

    def _colsq_len(self) -> int:
        return self.plan.info()["colsq_len"]

    def _device(self):
        return "cuda"

    def _stats(self, params, grads, momentum, lr, wd, mu, eps, stream):
        self.plan.rownorm_shard_stats(params, grads, momentum, lr, wd, self.colsq, mu, eps, stream)

    def _apply(self, params, grads, momentum, lr, wd, mu, eps, stream):
        self.plan.rownorm_shard_apply(params, grads, momentum, lr, wd, self.colsq, mu, eps, stream)

    def step(self, params, grads, momentum, lr: float, wd: float, mu: float = DEFAULT_MU, eps: float = 1e-8,
             stream=None):
        """One RowNorm step of this rank's shards: statistics, their sum over the ranks,
        the update."""
        import torch.distributed as dist
        self._stats(params, grads, momentum, lr, wd, mu, eps, stream)
        if dist.is_available() and dist.is_initialized() and dist.get_world_size(self.group) > 1:
            dist.all_reduce(self.colsq, op=dist.ReduceOp.SUM, group=self.group)
        self._apply(params, grads, momentum, lr, wd, mu, eps, stream)

    def close(self):
        if getattr(self, "plan", None) is not None and hasattr(self.plan, "close"):
            self.plan.close()
            self.plan = None


def select_precision(shapes, grad_dtype, params, grads, momentum, mu: float = DEFAULT_MU, tol: float = 1e-2,
                     sample: int = 4, candidates=(-1, 1), reference: int = 2, ns_steps: int = DEFAULT_NS_STEPS,
                     stream=None, **plan_opts):
    """Per-matrix precision levels for ``precision_of``, chosen on the caller's own data:
    DMuon's plan-time profiling per shape (technical summary sec. 2.3 and 2.4), with an
    accuracy check added because the candidates differ in their results.

    For every oriented shape, up to ``sample`` of its matrices run one NS step at the
    reference level (split level 2) and at each candidate level (< 0: the plain recipe,
    1: split recursion); a candidate passes when the O of every sampled matrix is within
    ``tol`` (relative Frobenius, ``muon_debug_update_error``) of the reference's O, and each
    shape takes the fastest passing candidate (step time of the sample, measured with CUDA
    events), else the reference.  The caller's tensors are not modified: the steps run on
    copies with lr = wd = 0.  Returns (levels, report): one level per matrix and, per shape,
    each candidate's error and milliseconds."""
    import torch
    shapes = [(int(m), int(n)) for m, n in shapes]
    groups = {}
    for i, (m, n) in enumerate(shapes):
        groups.setdefault((min(m, n), max(m, n)), []).append(i)
    picked = [i for key in groups for i in groups[key][:sample]]
    sub = [shapes[i] for i in picked]
    grads_s = [grads[i] for i in picked]
    levels_all = [reference] + [c for c in candidates if c != reference]

    def run(level, ref):
        plan = MuonPlan(sub, grad_dtype, keep_update=True, precision_of=[level] * len(sub), **plan_opts)
        try:
            W = [params[i].clone() for i in picked]
            M = [momentum[i].clone() for i in picked]
            plan.step(W, grads_s, M, 0.0, 0.0, mu, ns_steps, stream=stream)
            plan.sync(stream)
            if ref is None:
                out = [plan.debug_update(j) for j in range(len(sub))]
            else:
                out = [plan.debug_update_error(j, ref[j], stream) for j in range(len(sub))]
            s = torch.cuda.current_stream() if stream is None else stream
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(2):
                plan.step(W, grads_s, M, 0.0, 0.0, mu, ns_steps, stream=stream)
            e1.record(s)
            e1.synchronize()
            return out, e0.elapsed_time(e1) / 2
        finally:
            plan.close()

    ref_o, ref_ms = run(reference, None)
    errs, times = {reference: [0.0] * len(sub)}, {reference: ref_ms}
    for lv in levels_all[1:]:
        errs[lv], times[lv] = run(lv, ref_o)
    del ref_o
    levels = [reference] * len(shapes)
    report = {}
    for key, idx in groups.items():
        js = [picked.index(i) for i in idx[:sample]]
        rep = {lv: {"err": max(errs[lv][j] for j in js), "ms_sample": times[lv]} for lv in levels_all}
        ok = [lv for lv in levels_all if rep[lv]["err"] <= tol]
        chosen = min(ok, key=lambda lv: (times[lv], lv)) if ok else reference
        for i in idx:
            levels[i] = chosen
        report[key] = {"chosen": chosen, "candidates": rep}
    return levels, report


def measure_costs(shapes, grad_dtype: str = "bf16", sample: int = 4, reps: int = 2, ns_steps: int = DEFAULT_NS_STEPS,
                  **plan_opts):
    """Measured cost (milliseconds per matrix) of every matrix's NS step on this GPU, for
    ``partition_owners`` / ``DistributedMuon(costs=...)`` (DMuon technical summary sec. 2.3:
    the owner assignment balances measured per-shape times).  For every oriented shape, a
    plan over up to ``sample`` matrices of that shape (scratch tensors, seeded Gaussian
    values) is timed with CUDA events over ``reps`` steps after one warm-up; each matrix of
    the shape costs that time divided by the matrices timed."""
    import torch
    shapes = [(int(m), int(n)) for m, n in shapes]
    groups = {}
    for i, (m, n) in enumerate(shapes):
        groups.setdefault((min(m, n), max(m, n)), []).append(i)
    gdt = torch.bfloat16 if grad_dtype == "bf16" else torch.float32
    per_shape = {}
    for key, idx in groups.items():
        sub = [shapes[i] for i in idx[:sample]]
        gen = torch.Generator(device="cuda").manual_seed(len(per_shape) + 1)
        W = [torch.randn(s, device="cuda", generator=gen) * 0.02 for s in sub]
        G = [(torch.randn(s, device="cuda", generator=gen) * 1e-3).to(gdt) for s in sub]
        M = [torch.randn(s, device="cuda", generator=gen) * 1e-3 for s in sub]
        plan = MuonPlan(sub, grad_dtype, **plan_opts)
        try:
            plan.step(W, G, M, 0.02, 0.1, DEFAULT_MU, ns_steps)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                plan.step(W, G, M, 0.02, 0.1, DEFAULT_MU, ns_steps)
            e1.record()
            e1.synchronize()
            plan.sync()
            per_shape[key] = e0.elapsed_time(e1) / reps / len(sub)
        finally:
            plan.close()
        del W, G, M
    return [per_shape[(min(m, n), max(m, n))] for m, n in shapes]
