"""Benchmark of the Muon step on GB300.

Default: one GPU, the 28-layer Qwen2.5-7B-shaped set (196 matrices, 6.53e9
matrix parameters, bf16 grads, fp32 weights and momentum), NS5, 3 warm-up and
10 timed steps.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

With N > 1 (torchrun), the matrices are partitioned over the ranks, one owner
per matrix (DistributedMuon, longest processing time first); each rank steps its
own matrices and every owner then broadcasts its updated parameters to the other
ranks.  The work is fixed as N grows (strong scaling); the time is the max over
ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon step ms per param set; NS5 TFLOP/s as % of GB300 dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen7b_28l")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip muon_plan_tune (the plan's launch choices from its work estimate)")
    ap.add_argument("--full-symmetric", action="store_true",
                    help="symmetric r x r results stored whole (no lower-triangle storage)")
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="chunks of the e2e plan (host copies of one chunk overlap another's compute)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workspace-bytes", type=int, default=0,
                    help="cap on the plan's device workspace (the step then runs in chunks); 0: none")
    return ap.parse_args()


def gemm_source_sha(csrc: str) -> str:
    """First 16 hex digits of the SHA-256 of the tensor-core GEMM kernels' source
    (gemm.cu followed by gemm_common.cuh)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm.cu", "gemm_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def small_source_sha(csrc: str) -> str:
    """First 16 hex digits of the SHA-256 of the fused r <= 128 kernel's source
    (ns_small.cu followed by gemm_common.cuh)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("ns_small.cu", "gemm_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def small_traffic(workload: str):
    """DRAM bytes per launch of the fused r <= 128 kernel on the per-head workload,
    from the committed ncu summary (a smaller capture scaled by matrices); None
    unless it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "ns_small_kernel_qwen7b_heads_5l.md")
    csrc = os.path.join(ROOT, "matrix_orthogonalising_optimizer_muon_gb300", "csrc")
    if workload != "qwen7b_heads":
        return None
    try:
        vals = {}
        for line in open(path):
            if ":" in line and line.split(":")[0] in ("traffic_bytes_per_launch_qwen7b_heads", "small_source_sha256_16"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("small_source_sha256_16") != small_source_sha(csrc):
            return None
        return float(vals["traffic_bytes_per_launch_qwen7b_heads"])
    except (OSError, KeyError, ValueError):
        return None


def gemm_traffic(workload: str):
    """DRAM bytes per NS step of all tensor-core products, from the committed ncu
    summary; None unless it was taken on the current gemm kernel source."""
    path = os.path.join(ROOT, "profiles", "gemm_kernel_qwen7b_layer.md")
    csrc = os.path.join(ROOT, "matrix_orthogonalising_optimizer_muon_gb300", "csrc")
    if workload != "qwen7b_28l":
        return None
    try:
        vals = {}
        for line in open(path):
            if ":" in line and line.split(":")[0] in ("traffic_bytes_per_ns_step_qwen7b_28l", "gemm_source_sha256_16"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        sha = gemm_source_sha(csrc)
        if vals.get("gemm_source_sha256_16") != sha:
            return None
        return float(vals["traffic_bytes_per_ns_step_qwen7b_28l"])
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed plumbing
def dist_init(n_gpus):
    """(rank, world, local_rank); initialises torch.distributed when launched by torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host float over ranks (identity at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: int, world: int) -> int:
    """Sum of a host integer over ranks (identity at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


# ------------------------------------------------------------------ workload accounting
def algorithmic_ns_flops(shapes, ns_steps=5):
    """Tensor FLOPs of the Gram-form NS step, symmetric products counted at half:
    (SYRK r^2 c + final 2 r^2 c, bf16) and ((4J - 3) r x r products of r^3, fp16)."""
    rr = 0 if ns_steps == 0 else (1 if ns_steps == 1 else 4 * ns_steps - 3)
    rc = rrr = 0.0
    for m, n in shapes:
        r, c = min(m, n), max(m, n)
        rc += 3.0 * r * r * c
        rrr += rr * float(r) ** 3
    return rc, rrr


# ------------------------------------------------------------------ CPU oracle sample
def oracle_sample(shapes, grad_dtype, reps_per_bucket=1, seed=2):
    """Time the fp64 oracle (as it stands) on one matrix per distinct oriented shape
    and scale to the whole list.  Returns (estimated seconds per param set, detail)."""
    import numpy as np
    from oracle import muon_ref as R
    import workloads

    buckets = {}
    for i, (m, n) in enumerate(shapes):
        buckets.setdefault((min(m, n), max(m, n)), []).append(i)
    est, detail = 0.0, []
    for key, idx in sorted(buckets.items()):
        i = idx[0]
        m, n = shapes[i]
        w = workloads.gen_tensor((m, n), workloads.W_STD, workloads.seed_of(seed, 0, i, "W")).double().numpy()
        g = workloads.gen_tensor((m, n), workloads.G_STD, workloads.seed_of(seed, 0, i, "G"),
                                 dtype=grad_dtype).double().numpy()
        mm = workloads.gen_tensor((m, n), workloads.M_STD, workloads.seed_of(seed, 0, i, "M")).double().numpy()
        ts = []
        for _ in range(reps_per_bucket):
            t0 = time.perf_counter()
            R.muon_step(w, g, mm, workloads.LR, workloads.WD, workloads.MU, 5, "ns")
            ts.append(time.perf_counter() - t0)
        t = min(ts)
        est += t * len(idx)
        detail.append({"shape": [m, n], "count": len(idx), "s": round(t, 3)})
    return est, detail


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local):
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    import workloads

    wl = workloads.WORKLOADS[args.workload]
    shapes = list(wl.shapes)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()

    # ---- inputs resident in HBM (seeded on the device).  One gradient per matrix
    # serves every step (the step's cost does not depend on the gradient's values).
    # With N > 1 ranks each matrix has one owner (DistributedMuon: LPT over the
    # ranks); a rank keeps every parameter but only its own matrices' G and M.
    t0 = time.time()
    opt = None
    if world > 1:
        opt = lib.DistributedMuon(shapes, wl.grad_dtype, timing=True, workspace_bytes=args.workspace_bytes,
                                  full_symmetric=args.full_symmetric)
        owned = list(opt.owned)
        W = opt.allocate_params(dev)
        for i, (m, n) in enumerate(shapes):
            W[i].copy_(workloads.gen_tensor((m, n), workloads.W_STD, workloads.seed_of(wl.index, 0, i, "W"), dev))
    else:
        owned = list(range(len(shapes)))
        W = [workloads.gen_tensor((m, n), workloads.W_STD, workloads.seed_of(wl.index, 0, i, "W"), dev)
             for i, (m, n) in enumerate(shapes)]
    G, M = [None] * len(shapes), [None] * len(shapes)
    for i in owned:
        m, n = shapes[i]
        M[i] = workloads.gen_tensor((m, n), workloads.M_STD, workloads.seed_of(wl.index, 0, i, "M"), dev)
        G[i] = workloads.gen_tensor((m, n), workloads.G_STD, workloads.seed_of(wl.index, 0, i, "G"), dev,
                                    wl.grad_dtype)
    Wl, Gl, Ml = [W[i] for i in owned], [G[i] for i in owned], [M[i] for i in owned]
    if opt is not None:
        plan = opt.plan
    else:
        plan = lib.MuonPlan(shapes, wl.grad_dtype, timing=True, workspace_bytes=args.workspace_bytes,
                            full_symmetric=args.full_symmetric)
    torch.cuda.synchronize()
    setup_s = time.time() - t0
    lr, wd, mu = workloads.LR, workloads.WD, workloads.MU
    stream = torch.cuda.current_stream()
    if plan is not None:
        plan.bind(Wl, Gl, Ml)
        if not args.no_tune:   # plan-time tuning on the resident inputs (its steps precede the warm-up)
            plan.tune(Wl, Gl, Ml, workloads.LR, workloads.WD, workloads.MU, reps=2, stream=stream)

    def one_step(t):
        rownorm = bool(wl.rownorm_k and t % wl.rownorm_k != 0)
        if opt is not None:
            opt.step(W, G, M, lr, wd, mu, 5, "rownorm" if rownorm else "ns", eps=wl.eps, stream=stream)
        elif rownorm:
            plan.step_bound(lr, wd, mu, mode="rownorm", eps=wl.eps, stream=stream)
        else:
            plan.step_bound(lr, wd, mu, 5, "ns", stream=stream)

    for t in range(args.warmup):
        one_step(t)
    torch.cuda.synchronize()
    if plan is not None:
        plan.sync()
        try:
            plan.stage_times()               # drop the warm-up steps' event groups
        except lib.MuonError:
            pass

    # ---- timed region: K steps, CUDA events on the launching stream
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]   # end of each step
    launches = 0
    ev0.record(stream)
    for t in range(args.steps):
        one_step(args.warmup + t)
        ev_step[t].record(stream)
        launches += plan.info()["launches_last_step"] if plan is not None else 0
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if plan is not None:
        plan.sync()
        stage_ms, stage_fl = plan.stage_times()   # per-stage event times summed over the K steps
    else:
        stage_ms, stage_fl = [0.0] * 6, [0.0] * 3
    elapsed_ms = ev0.elapsed_time(ev1)
    ms_step = max_over_ranks(elapsed_ms / args.steps, world)
    per_step = [(ev0 if t == 0 else ev_step[t - 1]).elapsed_time(ev_step[t]) for t in range(args.steps)]
    return dict(wl=wl, shapes=shapes, local_shapes=[shapes[i] for i in owned], plan=plan, opt=opt,
                W=Wl, G=Gl, M=Ml, ms_step=ms_step, per_step=per_step, stage_ms=stage_ms,
                stage_fl=stage_fl, launches=launches, clocks=clk, peaks=peaks, peak_src=peak_src,
                setup_s=setup_s, one_step=one_step)


def run_e2e(res, args, copy_back=True):
    """Same step through the public API with host buffers (``muon_step_host``): every
    step copies the gradients host->device from pinned memory and the updated weights
    back device->host.  The plan runs in ``args.e2e_chunks`` chunks so that one chunk's
    copies overlap another chunk's compute; the stream waits for the last copy back.
    copy_back=False: the parameters stay on the device (as in training, where they live
    there) and each step's result read on the host is the plan's status word
    (``muon_sync``, 4 bytes)."""
    import torch
    import matrix_orthogonalising_optimizer_muon_gb300 as lib
    import workloads
    wl, shapes = res["wl"], res["local_shapes"]
    W, G, M = res["W"], res["G"], res["M"]
    if not shapes:
        return 0.0, 0, 0, 0, 0
    host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in G]
    host_w = [torch.empty(w.shape, dtype=w.dtype, pin_memory=True) for w in W] if copy_back else None
    for hg, g in zip(host_g, G):
        hg.copy_(g)
    plan = lib.MuonPlan(shapes, wl.grad_dtype, chunks=args.e2e_chunks)
    chunks = plan.info()["n_chunks"]
    lr, wd, mu = workloads.LR, workloads.WD, workloads.MU
    stream = torch.cuda.current_stream()

    def one(t):
        mode = "rownorm" if wl.rownorm_k and t % wl.rownorm_k != 0 else "ns"
        plan.step_host(W, G, M, host_g, host_w, lr, wd, mu, 5, mode, stream=stream)
        if not copy_back:
            plan.sync(stream)   # the step's status, read on the host

    one(0)   # warm-up: the plan's copy streams and events are created on first use
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 5))
    ev0.record(stream)
    for t in range(steps):
        one(args.warmup + t)
    ev1.record(stream)
    torch.cuda.synchronize()
    plan.sync()
    plan.close()
    h2d = sum(g.numel() * g.element_size() for g in G)
    d2h = sum(w.numel() * w.element_size() for w in W) if copy_back else 4
    return ev0.elapsed_time(ev1) / steps, h2d, d2h, steps, chunks


def report_ours(args, res, rank, world):
    wl, shapes = res["wl"], res["shapes"]
    peaks, src = res["peaks"], res["peak_src"]
    K = args.steps
    ms_step = res["ms_step"]
    st_ms, st_fl = res["stage_ms"], res["stage_fl"]
    n_ns = sum(1 for t in range(K) if not (wl.rownorm_k and (args.warmup + t) % wl.rownorm_k))
    n_rn = K - n_ns
    per_ns = [x / n_ns if n_ns else 0.0 for x in st_ms]
    gemm_ms = per_ns[1] + per_ns[2] + per_ns[3]
    gemm_fl = (st_fl[0] + st_fl[1] + st_fl[2]) / n_ns if n_ns else 0.0
    gbytes = 2 if wl.grad_dtype == "bf16" else 4
    local = res["local_shapes"]   # this rank's matrices (all of them on one GPU)
    small = [(m, n) for m, n in local if min(m, n) <= 128]
    small_bytes = sum(m * n * 12 for m, n in small)   # X read twice (bf16), W read + written (fp32)
    # The roofline object describes the step's dominant kernel: the tensor-core
    # products (algorithmic FLOPs over their event time, against the measured
    # sustained bf16 peak: they run inside a multi-second loop), or, when the fused
    # r <= 128 kernel dominates, its HBM traffic against the measured copy bandwidth.
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    roofline = None
    ns5 = {}
    if gemm_ms > 0 and gemm_fl > 0:
        achieved = gemm_fl / (gemm_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4), "traffic": gemm_traffic(wl.name),
                    "kernel": "gemm2_kernel: all tensor-core products of one NS5 step (SYRK, 17 r x r, final)",
                    "peak_note": "%s sustained dense bf16 (fp16 runs at the same rate)" % src}
        ns5 = {"ns5_tflops": round(achieved, 1),
               "ns5_frac_bf16_peak": round(achieved / peaks["bf16_tflops"], 4),
               "ns5_gemm_ms": round(gemm_ms, 3), "ns5_gemm_flops": gemm_fl}
    if per_ns[5] > 0 and small_bytes:
        gbs = small_bytes / (per_ns[5] * 1e-3) / 1e9
        ns5["fused_small_ms"] = round(per_ns[5], 3)
        ns5["fused_small_gbs"] = round(gbs, 1)
        # the fused kernel dominates when it takes longer than the products, or when the
        # products run beside it on the few CTA pairs left to them (a tensor roofline against
        # the whole GPU's peak would not describe them)
        beside = res["plan"] is not None and res["plan"].info().get("chain_clusters", 0) > 0
        if per_ns[5] > gemm_ms or beside:
            roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": small_traffic(wl.name),
                        "kernel": "ns_small_kernel: the whole NS5 step of the %d matrices with r <= 128 "
                                  "(12 B/elem: X read twice, W read and written)" % len(small),
                        "peak_note": "%s copy bandwidth" % src}
    line = {
        "metric": METRIC, "value": round(ms_step, 3), "unit": "ms", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": False,
        "scaling": "strong" if world > 1 else "weak", "vs_baseline": None,
        "dtype": "bf16/fp16 tensor (fp32 accumulate), fp32 elementwise",
        "data": "synthetic (seeded Gaussian, shapes of the workload)",
        "config": {"workload": wl.name, "matrices": len(shapes),
                   "params": int(sum(m * n for m, n in shapes)), "grad_dtype": wl.grad_dtype,
                   "ns_steps": 5, "rownorm_k": wl.rownorm_k,
                   "l2": "inputs larger than L2 (%.1f GB of W, G, M per step)" %
                         (sum(m * n for m, n in shapes) * (10 if wl.grad_dtype == "bf16" else 12) / 1e9),
                   "parallelism": ("owner partition over %d GPUs (LPT), one fp32 parameter broadcast per "
                                   "owner" % world) if world > 1 else "single GPU",
                   **({k: res["plan"].info()[k] for k in ("workspace_bytes", "lower_chunks", "tuned_candidates",
                                                          "chain_clusters")} if res["plan"] is not None else {}),
                   **({"rank0_matrices": len(local)} if world > 1 else {})},
        "stages_ms_per_ns_step": {"momentum_norm": round(per_ns[0], 3), "syrk": round(per_ns[1], 3),
                                  "ns_rxr": round(per_ns[2], 3), "final_apply": round(per_ns[3], 3),
                                  "fused_small": round(per_ns[5], 3)},
        # stage time x median SM clock = SM clock cycles (millions): comparable across runs whose
        # power-capped clocks differ, for the tensor-bound stages
        "stages_sm_mcycles_per_ns_step": ({k: round(v * res["clocks"]["sm_mhz"] / 1e3, 1) for k, v in
                                           (("syrk", per_ns[1]), ("ns_rxr", per_ns[2]), ("final_apply", per_ns[3]))}
                                          if (res["clocks"] or {}).get("sm_mhz") else None),
        "ms_per_step_median": round(statistics.median(res["per_step"]), 3),
        "ms_per_step_min": round(min(res["per_step"]), 3),
        "ns_steps_timed": n_ns,
        "roofline": roofline,
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if n_rn:
        line["rownorm_ms_per_rownorm_step"] = round(st_ms[4] / n_rn, 3)
        line["rownorm_steps_timed"] = n_rn
        rn_bytes = sum(m * n * (gbytes + 8 + 8) for m, n in local)   # G, M read + write, W read + write
        line["rownorm_step_gbs"] = round(rn_bytes / (st_ms[4] / n_rn * 1e-3) / 1e9, 1)
    line.update(ns5)
    if per_ns[0] > 0:
        mom_bytes = sum(m * n * (gbytes + 8 + 2) for m, n in local)
        line["momentum_kernel_gbs"] = round(mom_bytes / (per_ns[0] * 1e-3) / 1e9, 1)
        line["momentum_kernel_hbm_frac"] = round(line["momentum_kernel_gbs"] / peaks["hbm_gbs"], 4)
    return line


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args, rank, world):
    """The fp64 CPU oracle, as it stands, on the host cores.  Each step times the
    oracle on one matrix of one oriented shape (round robin over the shapes);
    the per-param-set time scales each shape's mean time by its count."""
    import workloads
    wl = workloads.WORKLOADS[args.workload]
    shapes = list(wl.shapes)
    if rank != 0:
        return None
    keys = sorted({(min(m, n), max(m, n)) for m, n in shapes})
    counts = {k: sum(1 for m, n in shapes if (min(m, n), max(m, n)) == k) for k in keys}
    first = {k: next(i for i, (m, n) in enumerate(shapes) if (min(m, n), max(m, n)) == k) for k in keys}
    times = {k: [] for k in keys}

    def sample(k):
        i = first[k]
        sub = [shapes[i]]
        t, _ = oracle_sample(sub, wl.grad_dtype, seed=wl.index)
        return t

    t0 = time.time()
    for s in range(args.warmup):
        sample(keys[s % len(keys)])
    for s in range(args.steps):
        k = keys[s % len(keys)]
        times[k].append(sample(k))
    for k in keys:                      # every shape timed at least once
        if not times[k]:
            times[k].append(sample(k))
    per_set = sum(counts[k] * statistics.mean(times[k]) for k in keys)
    ms = per_set * 1e3
    cores = os.cpu_count()
    return {
        "impl": "reference", "metric": METRIC, "value": round(ms, 1), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "matrices": len(shapes),
                   "params": int(sum(m * n for m, n in shapes))},
        "cpu_baseline": {"value": round(ms, 1), "unit": "ms", "cores": cores, "kind": "oracle",
                         "sample": "per step one matrix of one oriented shape (round robin over %d shapes), "
                                   "fp64 numpy direct NS5; scaled by the shape counts" % len(keys)},
        "e2e": {"value": round(ms, 1), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(time.time() - t0, 1),
    }


def main():
    args = parse_args()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    res = run_ours(args, rank, world, local)
    line = report_ours(args, res, rank, world)
    if not args.no_e2e:
        e2e_ms, h2d, d2h, nsteps, e2e_chunks = run_e2e(res, args)
        e2e_ms = max_over_ranks(e2e_ms, world)
        h2d, d2h = sum_over_ranks(h2d, world), sum_over_ranks(d2h, world)
        line["e2e"] = {"value": round(e2e_ms, 3), "unit": "ms", "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "steps": nsteps, "plan_chunks": e2e_chunks,
                       "what": "muon_step_host: grads host->device (pinned) and updated weights "
                               "device->host, overlapped chunk by chunk with the step" +
                               ("; each rank its own matrices, bytes summed over ranks" if world > 1 else "")}
        if world == 1:
            r_ms, r_h2d, r_d2h, r_steps, _ = run_e2e(res, args, copy_back=False)
            line["e2e_params_resident"] = {
                "value": round(r_ms, 3), "unit": "ms", "h2d_bytes_per_step": r_h2d, "d2h_bytes_per_step": r_d2h,
                "steps": r_steps, "what": "muon_step_host without the copy back: grads host->device (pinned), "
                                          "overlapped chunk by chunk; muon_sync reads the status every step"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, detail = oracle_sample(res["shapes"], res["wl"].grad_dtype, seed=res["wl"].index)
        line["cpu_baseline"] = {"value": round(t * 1e3, 1), "unit": "ms", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": "one matrix per oriented shape, fp64 numpy direct NS5, scaled by "
                                          "shape counts: %s" % json.dumps(detail)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
