"""The decode moment form's algebra, restated in numpy and held to the float64 oracle (no GPU).

The moment form (include/lla.h, lla_decode_ex) forms, for the new query,
    Cc = sum_j w_j (k_j - kbar) k_j^T,   Hc = sum_j w_j (k_j - kbar) v_j^T,
    r  = sum_j w_j (k_j - kbar),          nu = sum_j w_j v_j,
runs the centred CG with the operator p -> (Cc p - r (kbar.p))/omega + (lambda/omega) p, and ends with
    out = (nu - Hc^T x) / (omega - r.x),   rho = x / (1 + delta.x),   denom = omega / (1 + delta.x).
Every step is an identity of real arithmetic on the reading notes' Eqs. (6)-(8) (section 2.1), so in
float64 it must reproduce the oracle's exact solve at convergence and its centred CG at a fixed cap.
Planting each of these fails every case by orders of magnitude: the output moment untransposed
(Hc x), delta's sign, lambda not divided by omega, a wrong denominator.  The r terms are zero in
real arithmetic (they carry the rounding of kbar), and they make Cc's orientation immaterial too, so
only the GPU tests' fp32 gates exercise them.

The second test pins the design reason for centring on the exact kbar before the products: in fp32,
moments about the origin (Cu = sum_j w_j k_j k_j^T, then C = Cu - mu~ kbar^T) lose accuracy at second
order when the weighted keys share a component much larger than their spread.
"""
import math

import numpy as np
import pytest

from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
from oracle.lla_ref import lla_row, lla_row_deflated_cg


def moment_form(q, K, V, tau, lam, max_iters, tol, dt=np.float64, centred=True):
    q, K, V = (np.asarray(x, dtype=dt) for x in (q, K, V))
    s = (K @ q) * dt(tau)
    w = np.exp(s - s.max())
    omega = w.sum()
    kbar = (w @ K) / omega
    A = (K - kbar) * w[:, None]                    # w_j (k_j - kbar), the products' left operand
    Hc, r, nu = A.T @ V, A.sum(0), w @ V
    if centred:
        Cc = A.T @ K

        def apply_c(p):
            return Cc @ p - r * (kbar @ p)
    else:                                          # moments about the origin
        Cu, mu = (K * w[:, None]).T @ K, w @ K

        def apply_c(p):
            kp = kbar @ p
            return Cu @ p - mu * kp - kbar * (mu @ p - omega * kp)
    delta = kbar - q
    lam_n = dt(lam) / omega
    x = np.zeros_like(delta)
    res, p = delta.copy(), delta.copy()
    gamma = res @ res
    rn0 = math.sqrt(gamma)
    it = 0
    while it < max_iters and gamma > 0 and math.sqrt(gamma) > tol * rn0:
        cp = apply_c(p) / omega + lam_n * p
        pcp = p @ cp
        if not pcp > 0:
            break
        alpha = gamma / pcp
        x = x + alpha * p
        res = res - alpha * cp
        g2 = res @ res
        p = res + (g2 / gamma) * p
        gamma = g2
        it += 1
    g = 1 + delta @ x
    return {"out": (nu - Hc.T @ x) / (omega - r @ x), "rho": x / g, "denom": omega / g, "iters": it}


def _row(n, d, rising, seed=0):
    """The last row of a seeded LM-shaped sequence; with `rising`, key j moves along the query by
    3 (j // 64) / (tau |q|^2), so the logits rise by about 3 per 64 keys and the weighted keys share a
    component many times their spread."""
    w = workload("lm_bf16", B=1, H=1, n=n, d=d, tau=1.0 / math.sqrt(d), seed=seed)
    q, k, v = (t.double().numpy()[0, 0] for t in make_inputs(w))
    qi = q[n - 1]
    if rising:
        k = k + (3.0 * (np.arange(n) // 64))[:, None] * qi[None, :] / (w.tau * (qi @ qi))
    return w, qi, k, v


def _rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / np.abs(np.asarray(b)).max())


@pytest.mark.parametrize("rising", [False, True], ids=["plain", "rising"])
@pytest.mark.parametrize("n,d", [(300, 32), (700, 128)])
def test_moment_form_reproduces_the_oracle(n, d, rising):
    w, qi, K, V = _row(n, d, rising)
    exact = lla_row(qi, K, V, w.tau, w.lam)
    conv = moment_form(qi, K, V, w.tau, w.lam, 4 * d + 64, 1e-13)
    assert _rel(conv["out"], exact["out"]) < 1e-10
    assert _rel(conv["rho"], exact["rho"]) < 1e-10
    assert abs(conv["denom"] - exact["denom"]) < 1e-10 * exact["denom"]
    # the fixed cap: the same iteration, so the same iterate up to float64 rounding, which truncated
    # CG on the rising rows amplifies to ~1e-6
    capped = lla_row_deflated_cg(qi, K, V, w.tau, w.lam, 16, 0.0)
    mine = moment_form(qi, K, V, w.tau, w.lam, 16, 0.0)
    assert mine["iters"] == capped["iters"] == 16
    assert _rel(mine["out"], capped["out"]) < 1e-5
    assert _rel(mine["rho"], capped["rho"]) < 1e-5
    assert abs(mine["denom"] - capped["denom"]) < 1e-5 * capped["denom"]


@pytest.mark.parametrize("n,d", [(300, 32), (700, 128)])
def test_centring_keeps_fp32_rounding_first_order(n, d):
    w, qi, K, V = _row(n, d, rising=True)
    exact = lla_row(qi, K, V, w.tau, w.lam)
    rms = math.sqrt(float(np.mean(exact["rho"] ** 2)))
    err = {}
    for centred in (True, False):
        r = moment_form(qi, K, V, w.tau, w.lam, 4 * d + 64, 1e-6, dt=np.float32, centred=centred)
        err[centred] = float(np.abs(r["rho"] - exact["rho"]).max()) / rms
    assert err[True] < 2e-4
    assert err[False] > 5 * err[True], err
