"""Plain fp64 CPU oracle for one Muon optimizer step (test infrastructure only).

This module is TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py`` may import it.  The CUDA
library never calls it and shares no code with it.

Everything is float64 numpy, written to be read against the pages it follows:

* "Muon is Scalable for LLM Training" blog summary (taking-lying-flat, "Infra
  Optimizers"), Background section: update rule eq. (1), Nesterov input,
  Frobenius normalisation X0 = M/||M||_F, quintic Newton-Schulz eq. (2) with
  (a, b, c) = (3.4445, -4.7750, 2.0315); "Scaling Up Muon" section: decoupled
  weight decay eq. (3), Lemma 1 and the 0.2*sqrt(max(A, B)) scale of eq. (4).
* "Scaling Muon for Diffusion Transformers", section 2.1 (J_NS = 5, the finite
  map Phi_5, (1 - eta*lambda) W form), section 3.1 (orientation O(M): transpose
  when m > n; the polar factor; RowNorm R_eps(X)_i = X_i / max(||X_i||_2, eps)).
* "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead",
  technical summary section 2 "Gram Newton-Schulz": the recursion is run in the
  r x r Gram space G = X X^T.

Readings taken where the pages are silent:

* Nesterov: the NS (and RowNorm) input is U = mu*M_t + G_t with
  M_t = mu*M_{t-1} + G_t (no dampening); the stored state is M_t.
* What is Frobenius-normalised is U (the Nesterov input), exactly; ||U||_F = 0
  gives O = 0 (only weight decay acts).
* No transpose when m == n.
* RowNorm acts on the oriented U (not on X0), rows of the oriented matrix, i.e.
  original columns when m > n; its update uses the same scale 0.2*sqrt(max).

Parity pins: every function below is checked in ``tests/test_oracle.py``
against closed forms, invariants, a hand-written Jacobi SVD and brute force.
"""
from __future__ import annotations

import math
import numpy as np

# Newton-Schulz quintic coefficients, "Muon is Scalable" blog, Background, eq. (2).
NS_A = 3.4445
NS_B = -4.7750
NS_C = 2.0315
NS_COEFFS = (NS_A, NS_B, NS_C)
# Number of NS iterations, "Scaling Up Muon" (N = 5) and DiT paper sec. 2.1 (J_NS = 5).
NS_STEPS = 5
# Momentum coefficient, "Scaling Up Muon" (K. Jordan's setting, 0.95).
MU = 0.95
# RMS-matching factor of eq. (4), "Scaling Up Muon".
RMS_MATCH = 0.2


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------- elementwise
def momentum(m_prev, grad, mu: float = MU) -> np.ndarray:
    """M_t = mu * M_{t-1} + grad.  Blog eq. (1), first line."""
    return mu * _f64(m_prev) + _f64(grad)


def nesterov(m_t, grad, mu: float = MU) -> np.ndarray:
    """Nesterov NS input U = mu * M_t + grad.  Blog, Background (Nesterov-style momentum)."""
    return mu * _f64(m_t) + _f64(grad)


def update_scale(m: int, n: int) -> float:
    """s = 0.2 * sqrt(max(A, B)).  Blog eq. (4) with Lemma 1."""
    return RMS_MATCH * math.sqrt(max(m, n))


def apply_update(w, o, lr: float, wd: float, scale: float) -> np.ndarray:
    """W_t = W_{t-1} - lr * (scale * O_t + wd * W_{t-1}).  Blog eq. (3)/(4)."""
    w = _f64(w)
    return w - lr * (scale * _f64(o) + wd * w)


# ---------------------------------------------------------------- orientation
def orient(x) -> tuple[np.ndarray, bool]:
    """O(M): M if m <= n else M^T, so the result is r x c with r <= c.

    DiT paper sec. 3.1.  Returns (oriented matrix, transposed flag)."""
    x = _f64(x)
    if x.shape[0] <= x.shape[1]:
        return x, False
    return x.T, True


def deorient(x, transposed: bool) -> np.ndarray:
    """O^{-1}: maps the r x c result back to the stored m x n layout (sec. 3.1)."""
    return x.T if transposed else x


def frobenius_normalise(x) -> np.ndarray:
    """X0 = X / ||X||_F (blog, Background).  ||X||_F = 0 maps to the zero matrix."""
    x = _f64(x)
    nrm = math.sqrt(float(np.sum(x * x)))
    if nrm == 0.0:
        return np.zeros_like(x)
    return x / nrm


# ---------------------------------------------------------------- Newton-Schulz
def ns_direct(x0, steps: int = NS_STEPS, coeffs=NS_COEFFS) -> np.ndarray:
    """Quintic Newton-Schulz in the r x c space, blog eq. (2):

        X_k = a X_{k-1} + b (X X^T) X_{k-1} + c (X X^T)^2 X_{k-1},

    run for ``steps`` iterations from X_0 = x0 (already normalised)."""
    a, b, c = coeffs
    x = _f64(x0)
    for _ in range(steps):
        gram = x @ x.T
        x = a * x + b * (gram @ x) + c * (gram @ (gram @ x))
    return x


def ns_gram(x0, steps: int = NS_STEPS, coeffs=NS_COEFFS) -> np.ndarray:
    """The same iteration carried in the r x r Gram space (DMuon, Gram Newton-Schulz).

    With G_0 = X_0 X_0^T, each step is X_k = P_k X_{k-1} where
    P_k = a I + b G_{k-1} + c G_{k-1}^2.  Hence X_k = Q_k X_0 with
    Q_k = P_k Q_{k-1} (Q_0 = I), and G_k = X_k X_k^T = P_k G_{k-1} P_k^T,
    which equals G_{k-1} P_k^2 because every P_k is a polynomial in G_0 and so
    commutes with G_{k-1}.  Only r x r products are iterated; X_0 is touched
    twice (G_0 and the final Q_J X_0)."""
    a, b, c = coeffs
    x0 = _f64(x0)
    r = x0.shape[0]
    eye = np.eye(r)
    g = x0 @ x0.T
    q = eye.copy()
    for _ in range(steps):
        p = a * eye + b * g + c * (g @ g)
        q = p @ q
        g = g @ (p @ p)
    return q @ x0


def quintic(x: float, coeffs=NS_COEFFS) -> float:
    """f(x) = a x + b x^3 + c x^5 (blog, Background): the map NS applies to each singular value."""
    a, b, c = coeffs
    return a * x + b * x ** 3 + c * x ** 5


def quintic_iter(x: float, steps: int = NS_STEPS, coeffs=NS_COEFFS) -> float:
    for _ in range(steps):
        x = quintic(x, coeffs)
    return x


# ---------------------------------------------------------------- RowNorm
def rownorm(x, eps: float) -> np.ndarray:
    """R_eps(X)_{i:} = X_{i:} / max(||X_{i:}||_2, eps), i = 1..r.  DiT paper sec. 3.1."""
    x = _f64(x)
    norms = np.sqrt(np.sum(x * x, axis=1, keepdims=True))
    return x / np.maximum(norms, eps)


# ---------------------------------------------------------------- one step
def orthogonalised_update(u, steps: int = NS_STEPS, coeffs=NS_COEFFS,
                          form: str = "direct") -> np.ndarray:
    """O_t for a stored m x n Nesterov input U: orient, normalise, NS, de-orient."""
    xt, transposed = orient(u)
    x0 = frobenius_normalise(xt)
    if form == "direct":
        xj = ns_direct(x0, steps, coeffs)
    elif form == "gram":
        xj = ns_gram(x0, steps, coeffs)
    else:
        raise ValueError(form)
    return deorient(xj, transposed)


def rownorm_update(u, eps: float) -> np.ndarray:
    """RowNorm direction for a stored m x n U: orient, R_eps over oriented rows, de-orient."""
    xt, transposed = orient(u)
    return deorient(rownorm(xt, eps), transposed)


def muon_step(w, grad, m_prev, lr: float, wd: float, mu: float = MU,
              ns_steps: int = NS_STEPS, mode: str = "ns", eps: float = 1e-8,
              coeffs=NS_COEFFS, form: str = "direct"):
    """One Muon step on one matrix.  Returns (W_t, M_t, O_t) in float64.

    mode "ns":      O_t = NS_J(O(U)/||U||_F) mapped back (blog eqs. (1), (2), (4)).
    mode "rownorm": O_t = R_eps(O(U)) mapped back (DiT paper sec. 3, RowNorm step).
    Both use U = mu*M_t + G and W_t = W - lr*(0.2*sqrt(max(m, n))*O_t + wd*W)."""
    m_t = momentum(m_prev, grad, mu)
    u = nesterov(m_t, grad, mu)
    if mode == "ns":
        o = orthogonalised_update(u, ns_steps, coeffs, form)
    elif mode == "rownorm":
        o = rownorm_update(u, eps)
    else:
        raise ValueError(mode)
    m, n = u.shape
    w_t = apply_update(w, o, lr, wd, update_scale(m, n))
    return w_t, m_t, o


def schedule_mode(t: int, k: int) -> str:
    """Periodic RowNorm Muon (DiT paper sec. 3): full NS5 every K steps, RowNorm otherwise.

    Steps are counted from 0 and step t refreshes with NS iff t mod K == 0."""
    if k <= 0:
        raise ValueError("K must be positive")
    return "ns" if t % k == 0 else "rownorm"


# ---------------------------------------------------------------- Jacobi SVD
def jacobi_svd(a, tol: float = 1e-15, max_sweeps: int = 100):
    """Thin SVD by one-sided (Hestenes) Jacobi rotations, written out by hand.

    Returns (U, s, V) with A = U diag(s) V^T, s descending, U and V with
    orthonormal columns.  Used only to pin the NS oracle (singular-value map,
    cubic NS limit UV^T); it calls no LAPACK routine."""
    a = _f64(a)
    wide = a.shape[0] < a.shape[1]
    if wide:
        a = a.T
    m, n = a.shape
    w = a.copy()
    v = np.eye(n)
    for _ in range(max_sweeps):
        rotated = False
        for p in range(n - 1):
            for q in range(p + 1, n):
                alpha = float(np.dot(w[:, p], w[:, p]))
                beta = float(np.dot(w[:, q], w[:, q]))
                gamma = float(np.dot(w[:, p], w[:, q]))
                if abs(gamma) <= tol * math.sqrt(alpha * beta) or gamma == 0.0:
                    continue
                rotated = True
                zeta = (beta - alpha) / (2.0 * gamma)
                t = math.copysign(1.0, zeta) / (abs(zeta) + math.sqrt(1.0 + zeta * zeta))
                cs = 1.0 / math.sqrt(1.0 + t * t)
                sn = cs * t
                wp = w[:, p].copy()
                w[:, p] = cs * wp - sn * w[:, q]
                w[:, q] = sn * wp + cs * w[:, q]
                vp = v[:, p].copy()
                v[:, p] = cs * vp - sn * v[:, q]
                v[:, q] = sn * vp + cs * v[:, q]
        if not rotated:
            break
    s = np.sqrt(np.sum(w * w, axis=0))
    order = np.argsort(-s)
    s = s[order]
    v = v[:, order]
    w = w[:, order]
    u = np.zeros_like(w)
    for j in range(n):
        if s[j] > 0:
            u[:, j] = w[:, j] / s[j]
    if wide:
        return v, s, u
    return u, s, v
