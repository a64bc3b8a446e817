"""Pins for the float64 oracle, checked against facts it does not compute itself.

Every check here is a closed form, an invariant, a special case that reduces to a
textbook estimator, or brute force on tiny inputs (Local Linear Attention reading
notes, sections 2.1-2.2; Parallax summary; kernel-methods blog chapter 1).
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import lla_ref as O


def _rand(seed, n, d, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, d)) * scale, rng.standard_normal((n, d)) * scale,
            rng.standard_normal((n, d)))


CASES = [(0, 12, 4, 0.7, 0.3), (1, 16, 3, 1.3, 0.05), (2, 9, 4, 0.2, 2.0), (3, 16, 2, 2.5, 1e-3)]


@pytest.mark.parametrize("seed,n,d,tau,lam", CASES)
def test_closed_form_matches_brute_force_least_squares(seed, n, d, tau, lam):
    """Eqs. (6)-(8) closed form == direct minimisation of the section 2.1 objective.

    Rows i < d have a rank-deficient weighted scatter: lambda keeps the fit unique.
    """
    q, k, v = _rand(seed, n, d)
    for i in range(n):
        r = O.lla_row(q[i], k[: i + 1], v[: i + 1], tau, lam)
        b, W = O.brute_force_fit(q[i], k[: i + 1], v[: i + 1], r["w"], lam / 2.0)
        assert np.abs(r["out"] - b).max() <= 1e-10 * (1 + np.abs(b).max())


def test_brute_force_is_a_minimum():
    """The brute-force (b, W) is not beaten by any of 200 random perturbations."""
    q, k, v = _rand(7, 10, 3)
    i = 9
    w, _ = O.row_weights(q[i], k[: i + 1], 0.9)
    b, W = O.brute_force_fit(q[i], k[: i + 1], v[: i + 1], w, 0.25)
    f0 = O.ridge_objective(b, W, q[i], k[: i + 1], v[: i + 1], w, 0.25)
    rng = np.random.default_rng(0)
    for _ in range(200):
        eps = 10.0 ** rng.uniform(-6, -1)
        f1 = O.ridge_objective(b + eps * rng.standard_normal(3), W + eps * rng.standard_normal((3, 3)),
                               q[i], k[: i + 1], v[: i + 1], w, 0.25)
        assert f1 >= f0 - 1e-12


def test_printed_ridge_factor_reading():
    """The printed lambda||W||^2 corresponds to 2 lambda I, not Eq. (7)'s lambda I.

    Documents the reading: with ridge = lambda the brute force disagrees with the
    closed form; with ridge = lambda/2 it agrees (previous test).
    """
    q, k, v = _rand(0, 12, 4)
    i = 11
    r = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.7, 0.3)
    b, _ = O.brute_force_fit(q[i], k[: i + 1], v[: i + 1], r["w"], 0.3)
    assert np.abs(r["out"] - b).max() > 1e-4
    r2 = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.7, 0.6)
    assert np.abs(r2["out"] - b).max() < 1e-10


@pytest.mark.parametrize("seed,n,d,tau,lam", CASES)
def test_mixing_weights_sum_to_one_and_denominator_positive(seed, n, d, tau, lam):
    """sum_j s_ij = 1 and omega - mu^T rho > 0 (section 2.1 / Sec. 2.3)."""
    q, k, v = _rand(seed, n, d)
    neg = 0
    for i in range(n):
        r = O.lla_row(q[i], k[: i + 1], v[: i + 1], tau, lam)
        assert abs(r["s"].sum() - 1.0) < 1e-12
        assert r["denom"] > 0
        neg += int((r["s"] < 0).any())
    assert neg > 0 or lam > 1.0  # local-linear weights do go negative


@pytest.mark.parametrize("seed,n,d,tau,lam", CASES)
def test_eq9_linear_prediction_plus_local_residual(seed, n, d, tau, lam):
    """Eq. (9): b_i = W_i q_i + sum_j wbar_ij (v_j - W_i k_j)."""
    q, k, v = _rand(seed, n, d)
    for i in range(n):
        r = O.lla_row(q[i], k[: i + 1], v[: i + 1], tau, lam)
        W = O.slope_hat(q[i], k[: i + 1], v[: i + 1], r["w"], lam, r["out"])
        wbar = r["w"] / r["w"].sum()
        rhs = W @ q[i] + wbar @ (v[: i + 1] - k[: i + 1] @ W.T)
        assert np.abs(r["out"] - rhs).max() < 1e-10 * (1 + np.abs(rhs).max())


def test_eqs_10_12_split_equals_explicit_differences():
    """mu and Sigma through mu~ and Sigma~ (Eqs. (10)-(12)) equal the explicit-z forms."""
    q, k, _ = _rand(4, 30, 6)
    for i in [0, 5, 29]:
        w, _ = O.row_weights(q[i], k[: i + 1], 0.8)
        om, mu, Sig, _ = O.row_moments(q[i], k[: i + 1], w, 0.4)
        om2, mut, mu2, Sig2 = O.row_moments_split(q[i], k[: i + 1], w, 0.4)
        assert abs(om - om2) < 1e-12
        assert np.abs(mu - mu2).max() < 1e-12 * (1 + np.abs(mu).max())
        assert np.abs(Sig - Sig2).max() < 1e-11 * (1 + np.abs(Sig).max())
        assert np.abs(mut - w @ k[: i + 1]).max() < 1e-12


def test_lambda_to_infinity_is_softmax():
    """lambda -> infinity: rho -> 0 and s_ij -> w_ij / omega_i (Sec. 2.3)."""
    q, k, v = _rand(5, 40, 8)
    for i in [0, 1, 17, 39]:
        r = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.5, 1e12)
        sm = O.softmax_row(q[i], k[: i + 1], v[: i + 1], 0.5)
        assert np.abs(r["out"] - sm).max() < 1e-9
        assert np.abs(r["rho"]).max() < 1e-10


def test_softmax_is_normalised_kernel_average():
    """Nadaraya-Watson with exp(tau q.k) weights, written out with Fractions-free sums."""
    q, k, v = _rand(6, 5, 3)
    i = 4
    logits = [0.9 * float(q[i] @ k[j]) for j in range(i + 1)]
    ws = [math.exp(l) for l in logits]
    ref = sum(ws[j] * v[j] for j in range(i + 1)) / sum(ws)
    assert np.abs(O.softmax_row(q[i], k[: i + 1], v[: i + 1], 0.9) - ref).max() < 1e-13


@pytest.mark.parametrize("lam", [1e-3, 0.1, 1.0, 10.0])
def test_first_token_closed_form(lam):
    """i = 0: w = 1, z = k0 - q0, rho = z/(|z|^2+lambda), denom = lambda/(|z|^2+lambda), b = v0."""
    q, k, v = _rand(8, 1, 5)
    r = O.lla_row(q[0], k[:1], v[:1], 1.1, lam)
    z = k[0] - q[0]
    zz = z @ z
    # Sigma = z z^T + lambda I has condition (|z|^2 + lambda)/lambda: allow that much rounding
    cond = (zz + lam) / lam
    assert np.abs(r["rho"] - z / (zz + lam)).max() < 1e-15 * cond * np.abs(z).max()
    assert abs(r["denom"] - lam / (zz + lam)) < 1e-15 * cond
    assert np.abs(r["out"] - v[0]).max() < 1e-12


def test_one_dimensional_weighted_line_exact_rationals():
    """d = 1, three keys: the intercept of a weighted ridge line, in exact rationals.

    Textbook weighted least squares for y = b + W x with penalty (lambda/2) W^2 (the
    Eq. (7) reading): W = Sxy / (Sxx + lambda), b = ybar - W xbar with weighted
    means and centred sums.  Weights are supplied directly (no exp) so the whole
    expected value is an exact fraction.
    """
    x = [Fraction(1), Fraction(3), Fraction(-2)]          # z_j = k_j - q
    y = [Fraction(2), Fraction(-1), Fraction(5)]
    w = [Fraction(1), Fraction(1, 2), Fraction(1, 4)]
    lam = Fraction(1, 3)
    om = sum(w)
    xb = sum(a * b for a, b in zip(w, x)) / om
    yb = sum(a * b for a, b in zip(w, y)) / om
    sxx = sum(a * (b - xb) ** 2 for a, b in zip(w, x))
    sxy = sum(a * (b - xb) * (c - yb) for a, b, c in zip(w, x, y))
    W = sxy / (sxx + lam)
    b_exact = yb - W * xb
    # same data through the oracle's Eq. (8) pieces with explicit weights
    Z = np.array([[float(t)] for t in x])
    wf = np.array([float(t) for t in w])
    omega = wf.sum()
    mu = Z.T @ wf
    Sig = (Z * wf[:, None]).T @ Z + float(lam) * np.eye(1)
    rho = np.linalg.solve(Sig, mu)
    out, s, denom = O._output_from_rho(wf, Z, np.array([[float(t)] for t in y]), omega, mu, rho)
    assert abs(out[0] - float(b_exact)) < 1e-14


def test_affine_data_is_reproduced():
    """v_j = A k_j + c exactly affine, lambda ~ 0: the local line recovers A q + c."""
    rng = np.random.default_rng(9)
    n, d = 40, 4
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d))
    A = rng.standard_normal((d, d))
    c = rng.standard_normal(d)
    v = k @ A.T + c
    for i in [2 * d, 20, 39]:
        r = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.6, 1e-12)
        assert np.abs(r["out"] - (A @ q[i] + c)).max() < 1e-6


def test_constant_shift_and_linearity_in_values():
    """sum_j s_ij = 1 gives exact constant reproduction and shift equivariance; out is linear in V."""
    q, k, v = _rand(10, 25, 5)
    v2 = np.random.default_rng(11).standard_normal(v.shape)
    c = np.array([3.0, -1.0, 0.5, 2.0, -4.0])
    for i in [0, 7, 24]:
        base = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.8, 0.2)["out"]
        sh = O.lla_row(q[i], k[: i + 1], v[: i + 1] + c, 0.8, 0.2)["out"]
        const = O.lla_row(q[i], k[: i + 1], np.tile(c, (i + 1, 1)), 0.8, 0.2)["out"]
        lin = O.lla_row(q[i], k[: i + 1], 2 * v[: i + 1] - 3 * v2[: i + 1], 0.8, 0.2)["out"]
        b2 = O.lla_row(q[i], k[: i + 1], v2[: i + 1], 0.8, 0.2)["out"]
        assert np.abs(sh - (base + c)).max() < 1e-10
        assert np.abs(const - c).max() < 1e-10
        assert np.abs(lin - (2 * base - 3 * b2)).max() < 1e-10


def test_weight_normalisation_matters():
    """lambda is absolute: scaling every weight by e (a stale max) changes the output."""
    q, k, v = _rand(12, 20, 4)
    i = 19
    w, _ = O.row_weights(q[i], k[: i + 1], 0.8)
    Z = k[: i + 1] - q[i]

    def out_for(wt):
        om, mu, Sig, _ = O.row_moments(q[i], k[: i + 1], wt, 0.5)
        rho = np.linalg.solve(Sig, mu)
        return O._output_from_rho(wt, Z, v[: i + 1], om, mu, rho)[0]

    assert np.abs(out_for(w) - out_for(w * math.e)).max() > 1e-3
    assert w.max() == 1.0


def test_cg_solves_small_spd_exactly():
    """CG on a d x d SPD system reaches the solution in <= d steps (exact arithmetic).

    2 x 2 by hand: A = [[4, 1], [1, 3]], b = [1, 2] -> x = [1/11, 7/11].
    """
    x, it = O.cg_solve(np.array([[4.0, 1.0], [1.0, 3.0]]), np.array([1.0, 2.0]), 2, 0.0)
    assert it == 2
    assert np.abs(x - np.array([1 / 11, 7 / 11])).max() < 1e-14
    rng = np.random.default_rng(3)
    M = rng.standard_normal((8, 8))
    A = M @ M.T + 8 * np.eye(8)
    b = rng.standard_normal(8)
    x, it = O.cg_solve(A, b, 8, 0.0)
    assert np.abs(A @ x - b).max() < 1e-10
    x, it = O.cg_solve(A, b, 100, 1e-6)
    assert np.linalg.norm(A @ x - b) <= 1.01e-6 * np.linalg.norm(b) and it <= 8
    x, it = O.cg_solve(A, np.zeros(8), 10, 0.0)
    assert it == 0 and not x.any()


@pytest.mark.parametrize("seed,n,d,tau,lam", CASES)
def test_deflated_cg_converges_to_definition(seed, n, d, tau, lam):
    """Sherman-Morrison deflation is exact: run to convergence it equals the Cholesky solve."""
    q, k, v = _rand(seed, n, d)
    for i in range(n):
        a = O.lla_row(q[i], k[: i + 1], v[: i + 1], tau, lam)
        b = O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], tau, lam, 10 * d + 50, 0.0)
        assert np.abs(a["out"] - b["out"]).max() < 1e-9 * (1 + np.abs(a["out"]).max())
        assert np.abs(a["rho"] - b["rho"]).max() < 1e-9 * (1 + np.abs(a["rho"]).max())
        assert abs(a["denom"] - b["denom"]) < 1e-9 * a["denom"]
        assert abs(b["s"].sum() - 1.0) < 1e-12


def test_covariance_form_of_the_output():
    """Parallax form: b = vbar - eta Cov_vk rho for ANY rho, with denom = omega - mu.rho.

    Cov_vk = sum_j wbar_j (v_j - vbar)(k_j - kbar)^T, eta = omega / denom.  Holds
    exactly for any probe, so it also pins Eq. (8) away from the solve.
    """
    q, k, v = _rand(13, 30, 5)
    rng = np.random.default_rng(1)
    for i in [3, 29]:
        w, _ = O.row_weights(q[i], k[: i + 1], 0.7)
        om, mu, _, Z = O.row_moments(q[i], k[: i + 1], w, 0.3)
        wbar = w / om
        vb = wbar @ v[: i + 1]
        kb = wbar @ k[: i + 1]
        cov = ((v[: i + 1] - vb) * wbar[:, None]).T @ (k[: i + 1] - kb)
        for _ in range(5):
            rho = 0.05 * rng.standard_normal(5)
            out, _, denom = O._output_from_rho(w, Z, v[: i + 1], om, mu, rho)
            assert np.abs(out - (vb - (om / denom) * cov @ rho)).max() < 1e-12


def test_lla_ref_batched_layout_matches_rows():
    """lla_ref walks [B, H, n, d] row-major and honours an explicit row list."""
    rng = np.random.default_rng(14)
    q, k, v = (rng.standard_normal((2, 3, 6, 4)) for _ in range(3))
    out, rho, den = O.lla_ref(q, k, v, 0.5, 0.3)
    assert out.shape == (36, 4) and den.shape == (36,)
    r = O.lla_row(q[1, 2, 4], k[1, 2, :5], v[1, 2, :5], 0.5, 0.3)
    idx = (1 * 3 + 2) * 6 + 4
    assert np.abs(out[idx] - r["out"]).max() == 0.0
    o2, _, _ = O.lla_ref(q, k, v, 0.5, 0.3, rows=[(1, 2, 4), (0, 0, 0)])
    assert np.abs(o2[0] - r["out"]).max() == 0.0
    assert np.abs(o2[1] - v[0, 0, 0]).max() < 1e-12


def test_rounding_model_cg_matches_dense_cg_when_unperturbed():
    """The matrix-free centred CG used to model rounding: with u = 0 it takes the same steps as
    ``cg_solve`` on the dense centred matrix (same iteration count, same iterate to summation
    order), on a full-rank row and on a rank-deficient early row, capped and to tolerance."""
    q, k, v = _rand(16, 40, 8)
    rng = np.random.default_rng(0)
    for i, T, tol in [(39, 5, 0.0), (39, 200, 1e-10), (3, 6, 0.0), (3, 200, 1e-12)]:
        a = O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], 0.6, 0.2, T, tol)
        b = O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], 0.6, 0.2, T, tol, rounding=(0.0, rng))
        assert a["iters"] == b["iters"]
        assert np.abs(a["out"] - b["out"]).max() < 1e-10
        assert np.abs(a["rho"] - b["rho"]).max() < 1e-10 * max(1.0, np.abs(a["rho"]).max())


def test_rounding_model_converged_row_moves_by_about_u():
    """Run to convergence, a perturbation of relative size u in every product moves the solution
    by O(u kappa): tiny for u = 1e-9, visible but bounded for u = 1e-4, and zero difference for
    two runs with the same seed (the model is deterministic given its generator)."""
    q, k, v = _rand(17, 60, 4)
    i = 59
    ex = O.lla_row(q[i], k[: i + 1], v[: i + 1], 0.6, 0.5)["out"]
    run = lambda u, seed: O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], 0.6, 0.5, 400, 1e-13,
                                               rounding=(u, np.random.default_rng(seed)))["out"]
    assert np.abs(run(1e-9, 1) - ex).max() < 1e-6
    e4 = np.abs(run(1e-4, 1) - ex).max()
    assert 0.0 < e4 < 1e-1
    assert np.abs(run(1e-4, 5) - run(1e-4, 5)).max() == 0.0


def test_rounding_model_capped_rows_in_truncation_band_are_sensitive():
    """On an LM-shaped head at 16 iterations, a row in the truncation band (short prefix, CG far
    from converged) moves by far more than a converged late row under the same fp16-level
    perturbation: the spread the parity gate allows is a property of the row, not uniform."""
    from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
    w = workload("lm_bf16", B=1, H=1, n=700)
    q, k, v = (t.double().numpy()[0, 0] for t in make_inputs(w))
    def spread(i):
        base = O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], w.tau, w.lam, 16, 0.0)["out"]
        dev = [np.abs(O.lla_row_deflated_cg(q[i], k[: i + 1], v[: i + 1], w.tau, w.lam, 16, 0.0,
                                            rounding=(2.0 ** -11, np.random.default_rng(s)))["out"] - base).max()
               for s in range(2)]
        return max(dev)
    assert spread(100) > 10 * spread(690)


# --------------------------------------------------------------------------- Parallax form
def test_parallax_zero_probe_is_softmax():
    """Parallax page: with the probe projection set to zero the mechanism is exactly softmax."""
    q, k, v = _rand(21, 20, 4)
    for i in [0, 7, 19]:
        r = O.parallax_row(q[i], k[: i + 1], v[: i + 1], np.zeros(4), 0.9)
        assert np.abs(r["out"] - O.softmax_row(q[i], k[: i + 1], v[: i + 1], 0.9)).max() < 1e-14


def test_parallax_with_the_centred_solve_is_lla():
    """The Parallax rewrite of LLA: softmax minus Sigma_KV times the probe rho' = eta rho, where
    rho, denom come from the Cholesky solve of Eq. (7) and eta = omega / denom (the boundary
    factor the page drops by absorbing it into the probe)."""
    for seed, n, d, tau, lam in CASES:
        q, k, v = _rand(seed, n, d)
        for i in range(n):
            a = O.lla_row(q[i], k[: i + 1], v[: i + 1], tau, lam)
            probe = (a["omega"] / a["denom"]) * a["rho"]
            b = O.parallax_row(q[i], k[: i + 1], v[: i + 1], probe, tau)
            assert np.abs(a["out"] - b["out"]).max() < 1e-10 * (1 + np.abs(a["out"]).max())


def test_parallax_is_affine_in_the_probe():
    q, k, v = _rand(22, 25, 5)
    rng = np.random.default_rng(3)
    i = 24
    r1, r2 = rng.standard_normal(5), rng.standard_normal(5)
    f = lambda r: O.parallax_row(q[i], k[: i + 1], v[: i + 1], r, 0.6)["out"]
    lhs = f(2.0 * r1 - 0.5 * r2)
    rhs = f(np.zeros(5)) + 2.0 * (f(r1) - f(np.zeros(5))) - 0.5 * (f(r2) - f(np.zeros(5)))
    assert np.abs(lhs - rhs).max() < 1e-12


def test_parallax_uniform_weights_exact_rationals():
    """tau = 0: every prefix weight is 1, so the output is mean(v) - cov(v, k) rho with the
    population covariance, checked in exact rational arithmetic (d = 1)."""
    ks = [Fraction(x) for x in (3, -1, 4, 1, -5)]
    vs = [Fraction(x) for x in (2, 7, -1, 8, 2)]
    rho = Fraction(3, 7)
    K = np.array([[float(x)] for x in ks]); V = np.array([[float(x)] for x in vs])
    Q = np.zeros_like(K)
    for i in range(len(ks)):
        m = i + 1
        kb = sum(ks[: m]) / m
        vb = sum(vs[: m]) / m
        cov = sum((vs[j] - vb) * (ks[j] - kb) for j in range(m)) / m
        want = vb - cov * rho
        got = O.parallax_row(Q[i], K[: m], V[: m], np.array([float(rho)]), 0.0)["out"][0]
        assert abs(got - float(want)) < 1e-13


def test_parallax_ref_layout_matches_rows():
    rng = np.random.default_rng(23)
    q, k, v, r = (rng.standard_normal((2, 2, 5, 3)) for _ in range(4))
    out = O.parallax_ref(q, k, v, r, 0.4)
    assert out.shape == (20, 3)
    one = O.parallax_row(q[1, 0, 3], k[1, 0, :4], v[1, 0, :4], r[1, 0, 3], 0.4)["out"]
    assert np.abs(out[(1 * 2 + 0) * 5 + 3] - one).max() == 0.0


# --------------------------------------------------------------------------- backward
def _fd_grads(q, k, v, g, tau, lam, eps=1e-6):
    """Central finite differences of L = sum g . out over every input entry (float64)."""
    def L(q_, k_, v_):
        out, _, _ = O.lla_ref(q_, k_, v_, tau, lam)
        return float((out.reshape(g.shape) * g).sum())
    grads = []
    for which in range(3):
        base = [q, k, v]
        gr = np.zeros_like(base[which])
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            gr[idx] = (L(*plus) - L(*minus)) / (2 * eps)
        grads.append(gr)
    return grads


@pytest.mark.parametrize("seed,n,d,tau,lam", [(0, 7, 3, 0.8, 0.3), (1, 6, 4, 1.5, 0.05), (2, 5, 2, 0.3, 2.0)])
def test_gradient_matches_finite_differences(seed, n, d, tau, lam):
    """The derived backward equals central differences of the pinned forward on every entry,
    including the rank-deficient early rows (i < d) and the path through the row maximum."""
    rng = np.random.default_rng(seed)
    q, k, v, g = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    dq, dk, dv = O.lla_grad_ref(q, k, v, g, tau, lam)
    fq, fk, fv = _fd_grads(q, k, v, g, tau, lam)
    scale = max(np.abs(fq).max(), np.abs(fk).max(), np.abs(fv).max())
    for a, b in [(dq, fq), (dk, fk), (dv, fv)]:
        assert np.abs(a - b).max() <= 1e-6 * scale


def test_gradient_large_lambda_is_softmax_gradient():
    """lambda -> infinity: rho -> 0 and the backward tends to softmax attention's, whose closed
    form is dv_j = sum_i p_ij g_i and ds_ij = p_ij (g_i.v_j - g_i.out_i), dq_i = tau sum_j ds_ij k_j."""
    rng = np.random.default_rng(5)
    n, d, tau = 6, 3, 0.9
    q, k, v, g = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    dq, dk, dv = O.lla_grad_ref(q, k, v, g, tau, 1e12)
    Q, K, V, G = q[0, 0], k[0, 0], v[0, 0], g[0, 0]
    P = np.zeros((n, n))
    for i in range(n):
        e = np.exp(tau * K[: i + 1] @ Q[i] - (tau * K[: i + 1] @ Q[i]).max())
        P[i, : i + 1] = e / e.sum()
    out = P @ V
    dS = P * (G @ V.T - (G * out).sum(1, keepdims=True))
    assert np.abs(dv[0, 0] - P.T @ G).max() < 1e-9
    assert np.abs(dq[0, 0] - tau * dS @ K).max() < 1e-9
    assert np.abs(dk[0, 0] - tau * dS.T @ Q).max() < 1e-9


def test_gradient_is_linear_in_the_output_cotangent():
    rng = np.random.default_rng(6)
    q, k, v, g1, g2 = (rng.standard_normal((1, 1, 5, 3)) for _ in range(5))
    a = O.lla_grad_ref(q, k, v, g1, 0.7, 0.4)
    b = O.lla_grad_ref(q, k, v, g2, 0.7, 0.4)
    c = O.lla_grad_ref(q, k, v, 2.0 * g1 - g2, 0.7, 0.4)
    for x, y, z in zip(a, b, c):
        assert np.abs(z - (2.0 * x - y)).max() < 1e-10


def test_capped_gradient_converges_to_the_exact_gradient():
    """The iteration-capped backward (CG for rho' and for the adjoint) with a cap of d and a
    tight tolerance equals the finite-difference-pinned exact gradient."""
    rng = np.random.default_rng(7)
    q, k, v, g = (rng.standard_normal((1, 2, 9, 4)) for _ in range(4))
    a = O.lla_grad_ref(q, k, v, g, 0.6, 0.2)
    b = O.lla_grad_ref(q, k, v, g, 0.6, 0.2, cg=(40, 1e-14))
    for x, y in zip(a, b):
        assert np.abs(x - y).max() <= 1e-9 * np.abs(x).max()


def test_capped_gradient_with_no_iterations_is_softmax_gradient():
    """A cap of 0 leaves rho = u = 0: the backward of causal softmax attention (closed form)."""
    rng = np.random.default_rng(8)
    n, d, tau = 7, 3, 1.1
    q, k, v, g = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    dq, dk, dv = O.lla_grad_ref(q, k, v, g, tau, 0.5, cg=(0, 0.0))
    Q, K, V, G = q[0, 0], k[0, 0], v[0, 0], g[0, 0]
    P = np.zeros((n, n))
    for i in range(n):
        e = np.exp(tau * K[: i + 1] @ Q[i])
        P[i, : i + 1] = e / e.sum()
    dS = P * (G @ V.T - (G * (P @ V)).sum(1, keepdims=True))
    assert np.abs(dv[0, 0] - P.T @ G).max() < 1e-12
    assert np.abs(dq[0, 0] - tau * dS @ K).max() < 1e-12
    assert np.abs(dk[0, 0] - tau * dS.T @ Q).max() < 1e-12


def test_gradient_at_a_tie_takes_either_side():
    """Two equal top logits: the default takes the first index; the other index gives the other
    one-sided derivative, and the two differ only along the moved maximum."""
    rng = np.random.default_rng(9)
    d = 3
    K = rng.standard_normal((5, d))
    q = rng.standard_normal(d)
    K[1] = K[3] = 3.0 * q / np.linalg.norm(q)     # identical keys: tied logits, and the largest
    s = K @ q
    assert s[1] == s[3] == s.max() and int(np.argmax(s)) == 1
    V, g = rng.standard_normal((5, d)), rng.standard_normal(d)
    _, dq1, dK1, dV1 = O.lla_row_grad(q, K, V, g, 0.9, 0.4)
    _, dq3, dK3, dV3 = O.lla_row_grad(q, K, V, g, 0.9, 0.4, jm=3)
    assert np.abs(dV1 - dV3).max() < 1e-12
    # the maximum term moves from key 1 to key 3: dq equal (k_1 = k_3), dK swaps it between rows
    assert np.abs(dq1 - dq3).max() < 1e-12
    assert np.abs((dK1[1] + dK1[3]) - (dK3[1] + dK3[3])).max() < 1e-12
    keep = [0, 2, 4]
    assert np.abs(dK1[keep] - dK3[keep]).max() < 1e-12


def test_fp32_coefficient_error_behind_the_gates_model():
    """The parity gate's rounding model perturbs the fp32 path's per-pair CG coefficients at u = 2^-20
    (tests/parity_util.py).  That figure is the 90% quantile of the relative error a float32 evaluation
    of w_j (k_j.p - kbar.p) (two d-term dot products, each a sequential fp32 FMA chain) makes against
    float64 on LM-shaped rows; the median sits near 2^-22.  Re-measured here on a smaller sample."""
    from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
    w = workload("lm_bf16", B=1, H=2, n=1024)
    q, k, _ = (t.double().numpy()[0] for t in make_inputs(w))
    rng = np.random.default_rng(1)
    errs = []
    for h in range(w.H):
        for i in rng.integers(64, w.n, 8):
            K, qi = k[h, : i + 1], q[h, i]
            s = w.tau * K @ qi
            W = np.exp(s - s.max())
            kbar = (W / W.sum()) @ K
            p = rng.standard_normal(w.d)
            exact = W * ((K - kbar) @ p)
            K32, p32, kb32 = K.astype(np.float32), p.astype(np.float32), kbar.astype(np.float32)
            a = np.zeros(len(K), np.float32)
            kp = np.float32(0.0)
            for e in range(w.d):
                a = (a + K32[:, e] * p32[e]).astype(np.float32)
                kp = np.float32(kp + kb32[e] * p32[e])
            m32 = (W.astype(np.float32) * (a - kp)).astype(np.float64)
            errs.append(np.abs(m32 - exact) / np.abs(exact))
    e = np.concatenate(errs)
    assert 2.0 ** -24 < np.quantile(e, 0.5) < 2.0 ** -21
    assert 2.0 ** -22 < np.quantile(e, 0.9) < 2.0 ** -19
