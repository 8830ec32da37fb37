"""Pins for the fp64 oracle: each check ties it to something other than itself
(the pages' printed constants, closed forms, invariants, a hand-written Jacobi
SVD checked against LAPACK, brute-force loops on tiny inputs)."""
import math
import os

import numpy as np
import pytest

from oracle import muon_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


# ------------------------------------------------------------------ constants
def test_constants_match_pages():
    vals = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, value = line.split()[:2]
            vals[name] = float(value)
    assert R.NS_COEFFS == (vals["ns_a"], vals["ns_b"], vals["ns_c"])
    assert R.NS_STEPS == vals["ns_steps"]
    assert R.MU == vals["mu"]
    assert R.RMS_MATCH == vals["rms_match"]


def test_quintic_fixed_point_near_one():
    # blog, Background: f(x) = ax + bx^3 + cx^5 is chosen to have a fixed point near 1.
    # Fixed points solve c y^2 + b y + (a - 1) = 0 with y = x^2 (quadratic formula).
    a, b, c = R.NS_COEFFS
    disc = b * b - 4 * c * (a - 1)
    y = (-b - math.sqrt(disc)) / (2 * c)
    x = math.sqrt(y)
    assert 0.8 < x < 1.0
    assert abs(R.quintic(x) - x) < 1e-12
    # small singular values grow fast: slope a at 0
    assert abs(R.quintic(1e-6) / 1e-6 - a) < 1e-9


def test_quintic_range_on_gaussian_spectrum():
    # f^5 maps (0.02, 1] into a band around the fixed point; this is what keeps
    # RMS(O)*sqrt(c) near 1 (Lemma 1).
    xs = np.linspace(0.02, 1.0, 2001)
    ys = np.array([R.quintic_iter(x) for x in xs])
    assert ys.min() > 0.6 and ys.max() < 1.2


# ------------------------------------------------------------------ elementwise
def test_momentum_geometric_series():
    # M_0 = 0 (blog: momentum starts at zero); constant gradient g for T steps:
    # M_T = g (1 - mu^T) / (1 - mu).
    g = rng(1).standard_normal((3, 5))
    m = np.zeros_like(g)
    mu, T = 0.95, 37
    for _ in range(T):
        m = R.momentum(m, g, mu)
    np.testing.assert_allclose(m, g * (1 - mu ** T) / (1 - mu), rtol=1e-12)


def test_nesterov_first_step_and_limit():
    g = rng(2).standard_normal((4, 6))
    mu = 0.95
    m1 = R.momentum(np.zeros_like(g), g, mu)
    np.testing.assert_allclose(R.nesterov(m1, g, mu), (1 + mu) * g, rtol=1e-15)
    m = np.zeros_like(g)
    for _ in range(2000):
        m = R.momentum(m, g, mu)
    np.testing.assert_allclose(R.nesterov(m, g, mu), g / (1 - mu), rtol=1e-12)


def test_apply_matches_dit_paper_form():
    # DiT paper sec. 2.1 writes the same update as W' = (1 - lr*wd) W - lr*s*P.
    w = rng(3).standard_normal((5, 7))
    o = rng(4).standard_normal((5, 7))
    lr, wd, s = 0.02, 0.1, R.update_scale(5, 7)
    np.testing.assert_allclose(R.apply_update(w, o, lr, wd, s),
                               (1 - lr * wd) * w - lr * s * o, rtol=1e-14)
    np.testing.assert_array_equal(R.apply_update(w, o, 0.0, wd, s), w)


def test_update_scale_lemma1():
    # Lemma 1: a full-rank [A, B] matrix's exact orthogonalised update has RMS
    # 1/sqrt(max(A, B)); scaled by 0.2*sqrt(max) it has RMS 0.2 for every shape.
    for shape in [(4, 9), (9, 4), (6, 6), (1, 8)]:
        u, s, v = R.jacobi_svd(rng(5).standard_normal(shape))
        polar = u @ v.T
        rms = math.sqrt(float(np.mean(polar ** 2)))
        assert abs(rms - 1 / math.sqrt(max(shape))) < 1e-12
        assert abs(R.update_scale(*shape) * rms - 0.2) < 1e-12


# ------------------------------------------------------------------ orientation / norm
def test_orient():
    x = rng(6).standard_normal((7, 3))
    xt, tr = R.orient(x)
    assert tr and xt.shape == (3, 7)
    np.testing.assert_array_equal(R.deorient(xt, tr), x)
    sq = rng(7).standard_normal((4, 4))
    assert R.orient(sq)[1] is False
    wide = rng(8).standard_normal((2, 9))
    assert R.orient(wide)[1] is False


def test_frobenius_normalise():
    x = rng(9).standard_normal((3, 8)) * 1e-3
    x0 = R.frobenius_normalise(x)
    assert abs(np.sum(x0 ** 2) - 1) < 1e-14
    np.testing.assert_array_equal(R.frobenius_normalise(np.zeros((2, 3))), np.zeros((2, 3)))


# ------------------------------------------------------------------ Jacobi SVD
@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (5, 5), (1, 6), (12, 3)])
def test_jacobi_svd_against_lapack(shape):
    a = rng(10).standard_normal(shape)
    u, s, v = R.jacobi_svd(a)
    r = min(shape)
    assert u.shape == (shape[0], r) and v.shape == (shape[1], r)
    np.testing.assert_allclose(u @ np.diag(s) @ v.T, a, atol=1e-13)
    np.testing.assert_allclose(u.T @ u, np.eye(r), atol=1e-13)
    np.testing.assert_allclose(v.T @ v, np.eye(r), atol=1e-13)
    np.testing.assert_allclose(s, np.linalg.svd(a, compute_uv=False), rtol=1e-13)


# ------------------------------------------------------------------ Newton-Schulz
@pytest.mark.parametrize("shape", [(8, 16), (16, 8)])
def test_ns5_is_quintic_on_singular_values(shape):
    # Blog, Background: NS keeps the singular vectors and applies f five times
    # to sigma_i / ||U||_F.  Checked through the full orient/normalise path.
    u_in = rng(11).standard_normal(shape)
    uu, s, vv = R.jacobi_svd(u_in)
    fro = math.sqrt(float(np.sum(s ** 2)))
    expect = uu @ np.diag([R.quintic_iter(x / fro) for x in s]) @ vv.T
    got = R.orthogonalised_update(u_in, 5)
    np.testing.assert_allclose(got, expect, atol=1e-12)


def test_rank1_closed_form():
    # U = x y^T has one singular value; O = f^5(1) * xhat yhat^T.
    x, y = rng(12).standard_normal(6), rng(13).standard_normal(11)
    f = 1.0
    a, b, c = R.NS_COEFFS
    for _ in range(5):
        f = a * f + b * f ** 3 + c * f ** 5
    assert abs((a + b + c) - 0.701) < 1e-15        # f(1) = a + b + c
    o = R.orthogonalised_update(np.outer(x, y), 5)
    np.testing.assert_allclose(o, f * np.outer(x / np.linalg.norm(x), y / np.linalg.norm(y)),
                               atol=1e-13)
    # the committed fixture
    with open(os.path.join(GOLDEN, "rank1_f5.txt")) as fh:
        stored = float([l for l in fh if not l.startswith("#")][0])
    assert abs(stored - f) < 1e-15


def test_cubic_ns_converges_to_polar():
    # Blog, Background: the iteration approximates (M M^T)^{-1/2} M = U V^T.
    # With (a, b, c) = (1.5, -0.5, 0) it is the classical cubic NS; 50 steps
    # from a well-conditioned start reach U V^T to rounding.
    a_in = rng(14).standard_normal((8, 16))
    uu, s, vv = R.jacobi_svd(a_in)
    assert s[-1] / np.linalg.norm(s) > 0.05
    got = R.orthogonalised_update(a_in, 50, coeffs=(1.5, -0.5, 0.0))
    np.testing.assert_allclose(got, uu @ vv.T, atol=1e-12)


@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (12, 12), (5, 40), (33, 70)])
def test_gram_form_equals_direct(shape):
    # DMuon's Gram-space recursion reaches the same X_J as eq. (2) in exact arithmetic.
    u_in = rng(15).standard_normal(shape)
    d = R.orthogonalised_update(u_in, 5, form="direct")
    g = R.orthogonalised_update(u_in, 5, form="gram")
    assert rel(g, d) < 1e-10


def test_ns_invariances():
    u_in = rng(16).standard_normal((6, 10))
    o = R.orthogonalised_update(u_in)
    # scale invariance (Frobenius normalisation)
    np.testing.assert_allclose(R.orthogonalised_update(3.7e-4 * u_in), o, atol=1e-13)
    # orthogonal equivariance NS(Q U R) = Q NS(U) R
    q, _ = np.linalg.qr(rng(17).standard_normal((6, 6)))
    r, _ = np.linalg.qr(rng(18).standard_normal((10, 10)))
    np.testing.assert_allclose(R.orthogonalised_update(q @ u_in @ r), q @ o @ r, atol=1e-12)
    # transpose equivariance (exercises orientation)
    np.testing.assert_allclose(R.orthogonalised_update(u_in.T), o.T, atol=1e-13)
    # zero iterations: X0 itself
    np.testing.assert_allclose(R.orthogonalised_update(u_in, 0), u_in / np.linalg.norm(u_in),
                               atol=1e-15)
    # zero input: zero update
    np.testing.assert_array_equal(R.orthogonalised_update(np.zeros((3, 4))), np.zeros((3, 4)))


def test_diagonal_input():
    d = np.array([3.0, -1.0, 0.5, 0.0])
    x = np.zeros((4, 7))
    x[np.arange(4), np.arange(4)] = d
    fro = np.linalg.norm(d)
    got = R.orthogonalised_update(x)
    expect = np.zeros_like(x)
    for i, di in enumerate(d):
        expect[i, i] = math.copysign(R.quintic_iter(abs(di) / fro), di)
    np.testing.assert_allclose(got, expect, atol=1e-14)


# ------------------------------------------------------------------ RowNorm
def brute_rownorm(x, eps):
    out = np.zeros_like(x)
    for i in range(x.shape[0]):
        s = 0.0
        for j in range(x.shape[1]):
            s += x[i, j] * x[i, j]
        d = max(math.sqrt(s), eps)
        for j in range(x.shape[1]):
            out[i, j] = x[i, j] / d
    return out


def test_rownorm_brute_force_and_unit_rows():
    x = rng(19).standard_normal((5, 9))
    x[2] *= 1e-12           # below eps: scaled by 1/eps, not normalised
    x[3] = 0.0              # zero row stays zero
    eps = 1e-8
    got = R.rownorm(x, eps)
    np.testing.assert_allclose(got, brute_rownorm(x, eps), rtol=1e-14, atol=0)
    norms = np.linalg.norm(got, axis=1)
    np.testing.assert_allclose(norms[[0, 1, 4]], 1.0, rtol=1e-14)
    np.testing.assert_allclose(got[2], x[2] / eps, rtol=1e-14)
    assert np.all(got[3] == 0)
    # RMS of a unit-row r x c matrix is 1/sqrt(c): same as Lemma 1's 1/sqrt(max)
    y = R.rownorm(rng(20).standard_normal((4, 25)), eps)
    assert abs(math.sqrt(np.mean(y ** 2)) - 1 / 5) < 1e-14


def test_rownorm_update_uses_oriented_rows():
    # m > n: the oriented rows are the stored columns.
    x = rng(21).standard_normal((9, 4))
    got = R.rownorm_update(x, 1e-8)
    np.testing.assert_allclose(np.linalg.norm(got, axis=0), 1.0, rtol=1e-14)
    np.testing.assert_allclose(got, brute_rownorm(x.T, 1e-8).T, rtol=1e-14)
    y = rng(22).standard_normal((4, 9))
    np.testing.assert_allclose(R.rownorm_update(y, 1e-8), brute_rownorm(y, 1e-8), rtol=1e-14)


# ------------------------------------------------------------------ full step
@pytest.mark.parametrize("mode", ["ns", "rownorm"])
def test_step_transpose_equivariance(mode):
    w, g, m = (rng(s).standard_normal((6, 11)) for s in (23, 24, 25))
    a = R.muon_step(w, g, m, 0.02, 0.1, mode=mode)
    b = R.muon_step(w.T, g.T, m.T, 0.02, 0.1, mode=mode)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y.T, atol=1e-14)


def test_step_composition():
    # One step = momentum, Nesterov, orthogonalised update, eq. (4), each
    # checked against its own closed form above; here the wiring.
    w, g, m = (rng(s).standard_normal((5, 8)) for s in (26, 27, 28))
    lr, wd, mu = 0.02, 0.1, 0.95
    w1, m1, o1 = R.muon_step(w, g, m, lr, wd, mu)
    np.testing.assert_allclose(m1, mu * m + g, rtol=1e-15)
    u = mu * m1 + g
    np.testing.assert_allclose(o1, R.orthogonalised_update(u), rtol=1e-15)
    np.testing.assert_allclose(w1, w - lr * (0.2 * math.sqrt(8) * o1 + wd * w), rtol=1e-15)
    # ns_steps = 0: the update is X0
    _, _, o0 = R.muon_step(w, g, m, lr, wd, mu, ns_steps=0)
    np.testing.assert_allclose(o0, u / np.linalg.norm(u), rtol=1e-14)
    # zero Nesterov input: only weight decay acts
    wz, _, oz = R.muon_step(w, np.zeros_like(g), np.zeros_like(m), lr, wd, mu)
    assert np.all(oz == 0)
    np.testing.assert_allclose(wz, (1 - lr * wd) * w, rtol=1e-15)


def test_schedule():
    # DiT paper sec. 3: NS5 every K steps; with K = 4 over 8 steps, NS at 0 and 4.
    modes = [R.schedule_mode(t, 4) for t in range(8)]
    assert [t for t, m in enumerate(modes) if m == "ns"] == [0, 4]
    assert R.schedule_mode(5, 1) == "ns"


# ------------------------------------------------------------------ planted mistakes
def _mutant_direct(kind):
    def ns(x0, steps=5, coeffs=R.NS_COEFFS):
        a, b, c = coeffs
        x = np.asarray(x0, float)
        for _ in range(steps):
            gram = x @ x.T
            if kind == "drop_c":
                x = a * x + b * (gram @ x)
            elif kind == "sign_b":
                x = a * x - b * (gram @ x) + c * (gram @ (gram @ x))
            elif kind == "gram_once_in_c":
                x = a * x + b * (gram @ x) + c * (gram @ x)
            elif kind == "wrong_side":       # X (X X^T) instead of (X X^T) X
                x = a * x + b * (x @ gram) + c * (x @ gram @ gram)
        return x
    return ns


def _mutant_gram(x0, steps=5, coeffs=R.NS_COEFFS):
    a, b, c = coeffs
    x0 = np.asarray(x0, float)
    eye = np.eye(x0.shape[0])
    g, q = x0 @ x0.T, eye
    for _ in range(steps):
        p = a * eye + b * g + c * (g @ g)
        q = p @ q
        g = g @ p                            # should be g @ p @ p
    return q @ x0


@pytest.mark.parametrize("kind", ["drop_c", "sign_b", "gram_once_in_c", "wrong_side"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    """A plausible mistake planted in the oracle (on the CPU) fails the SVD pin."""
    monkeypatch.setattr(R, "ns_direct", _mutant_direct(kind))
    u_in = rng(29).standard_normal((12, 12))
    uu, s, vv = R.jacobi_svd(u_in)
    fro = np.linalg.norm(s)
    expect = uu @ np.diag([R.quintic_iter(x / fro) for x in s]) @ vv.T
    got = R.orthogonalised_update(u_in, 5)
    assert np.max(np.abs(got - expect)) > 1e-3


def test_planted_gram_mistake_is_caught(monkeypatch):
    u_in = rng(30).standard_normal((8, 16))
    d = R.orthogonalised_update(u_in, 5, form="direct")
    monkeypatch.setattr(R, "ns_gram", _mutant_gram)
    assert rel(R.orthogonalised_update(u_in, 5, form="gram"), d) > 1e-3
