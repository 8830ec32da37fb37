"""Seeded synthetic inputs for the Muon step: shapes of the benchmark workloads
and deterministic generators.  Shared by the tests, the oracle side and the
bench; holds none of the method's arithmetic (no momentum, normalisation,
Newton-Schulz or update code lives here).

Workloads (shapes as stored, row-major m x n):

* ``single``: one 256 x 1024 fp32 matrix (W, G, M all fp32).
* ``qwen7b_layer``: one Qwen2.5-7B decoder layer (hidden 3584, 28 q heads,
  4 kv heads, head_dim 128, FFN 18944): q, k, v, o, gate, up, down.
* ``qwen7b_28l``: the same layer repeated 28 times (196 matrices).
* ``qwen7b_heads``: per-head split, 28 x (28 q + 4 k + 4 v) 128 x 3584
  matrices plus 28 transposed-aspect 3584 x 512 matrices.
* ``dit1p3b``: 28 DiT blocks at hidden 2048: qkv 6144x2048, attn-out 2048x2048,
  mlp-in 8192x2048, mlp-out 2048x8192, adaLN 12288x2048 (periodic RowNorm, K=4).
* ``dit_block``: one of those blocks (0.75 GB of W, G, M: still above L2), the
  small case used to profile the RowNorm kernels.
* ``qwen7b_heads_5l``: five layers of the per-head split (180 matrices 128 x 3584
  and five 3584 x 512; 0.9 GB of W, G, M: above L2, and enough matrices to fill
  every SM), the small case used to profile the fused r <= 128 kernel.

Values: W ~ N(0, 0.02^2), G ~ N(0, 1e-3^2), M ~ N(0, 1e-3^2); G is bf16 except
in ``single``.  Each tensor gets its own seed from (workload, step, matrix, kind).
"""
from __future__ import annotations

from dataclasses import dataclass

HIDDEN_7B, FFN_7B, KV_7B = 3584, 18944, 512
HIDDEN_DIT = 2048

W_STD, G_STD, M_STD = 0.02, 1e-3, 1e-3
LR, WD, MU = 0.02, 0.1, 0.95


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple          # ((m, n), ...) as stored
    grad_dtype: str        # "f32" or "bf16"
    index: int             # base seed
    steps: int = 1
    rownorm_k: int = 0     # 0: NS every step; K > 0: NS iff t % K == 0
    eps: float = 1e-8


def _qwen_layer():
    h, f, kv = HIDDEN_7B, FFN_7B, KV_7B
    return ((h, h), (kv, h), (kv, h), (h, h), (f, h), (f, h), (h, f))


def _qwen_heads():
    one = ((128, HIDDEN_7B),) * (28 + 4 + 4)
    return one * 28 + ((HIDDEN_7B, 512),) * 28


def _qwen_heads_layers(n):
    return (((128, HIDDEN_7B),) * (28 + 4 + 4) + ((HIDDEN_7B, 512),)) * n


def _dit_block():
    h = HIDDEN_DIT
    return ((3 * h, h), (h, h), (4 * h, h), (h, 4 * h), (6 * h, h))


WORKLOADS = {
    "single": Workload("single", ((256, 1024),), "f32", 0),
    "qwen7b_layer": Workload("qwen7b_layer", _qwen_layer(), "bf16", 1),
    "qwen7b_28l": Workload("qwen7b_28l", _qwen_layer() * 28, "bf16", 2, steps=10),
    "qwen7b_heads": Workload("qwen7b_heads", _qwen_heads(), "bf16", 3),
    "dit1p3b": Workload("dit1p3b", _dit_block() * 28, "bf16", 4, steps=8, rownorm_k=4),
    "dit_block": Workload("dit_block", _dit_block(), "bf16", 5, steps=8, rownorm_k=4),
    "qwen7b_heads_5l": Workload("qwen7b_heads_5l", _qwen_heads_layers(5), "bf16", 6),
}


def seed_of(workload_index: int, step: int, matrix: int, kind: str) -> int:
    """Deterministic 63-bit seed for one tensor; kind in {"W", "G", "M"}."""
    k = {"W": 1, "G": 2, "M": 3}[kind]
    h = 0x9E3779B97F4A7C15
    for v in (workload_index, step, matrix, k):
        h ^= (v + 0x9E3779B97F4A7C15 + ((h << 6) & 0xFFFFFFFFFFFFFFFF) + (h >> 2)) & 0xFFFFFFFFFFFFFFFF
        h &= 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def gen_tensor(shape, std: float, seed: int, device="cpu", dtype="f32"):
    """N(0, std^2) tensor from torch's Philox/MT generator on ``device``, cast to dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t


def matrix_inputs(wl: Workload, step: int, idx: int, device="cpu"):
    """(W, G, M) torch tensors for matrix ``idx`` of ``wl`` at ``step``.

    W and M are the step-0 state; later steps of a multi-step run carry W and M
    forward and only draw a fresh G."""
    m, n = wl.shapes[idx]
    w = gen_tensor((m, n), W_STD, seed_of(wl.index, 0, idx, "W"), device)
    g = gen_tensor((m, n), G_STD, seed_of(wl.index, step, idx, "G"), device, wl.grad_dtype)
    mom = gen_tensor((m, n), M_STD, seed_of(wl.index, 0, idx, "M"), device)
    return w, g, mom


def grad_input(wl: Workload, step: int, idx: int, device="cpu"):
    m, n = wl.shapes[idx]
    return gen_tensor((m, n), G_STD, seed_of(wl.index, step, idx, "G"), device, wl.grad_dtype)


def numpy_matrix(shape, seed: int, std: float = 1.0):
    """Small numpy N(0, std^2) matrix for CPU-only tests."""
    import numpy as np
    return np.random.default_rng(seed).standard_normal(shape) * std
