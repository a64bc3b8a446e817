"""Plain float64 CPU oracle for the causal Local Linear Attention (LLA) forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
call it.  It shares no code with the CUDA path.

It is the plain definition written out, one query at a time, in float64:

* Local Linear Attention reading notes, section 2.1 ("one intercept per query"),
  Eqs. (6)-(8): for query i, with z_ij = k_j - q_i and kernel weights w_ij over
  the causal prefix j <= i,
      omega_i = sum_j w_ij,   mu_i = sum_j w_ij z_ij,
      Sigma_i = sum_j w_ij z_ij z_ij^T + lambda I,   rho_i = Sigma_i^{-1} mu_i,
      s_ij    = w_ij (1 - z_ij^T rho_i) / (omega_i - mu_i^T rho_i),
      b_i     = sum_j s_ij v_j.
  Every z_ij is formed explicitly and Sigma_i is built densely and factorised by
  Cholesky (the "naive" form of section 2.2, per row, never used on the GPU).
* The kernel weight is the dot-product exponential with the row maximum
  subtracted, w_ij = exp(tau q_i.k_j - max_{l<=i} tau q_i.k_l): the reading notes
  section 2.2 / Algorithm 1 accumulate the moments "with an online maximum",
  and the largest weight of a row is therefore 1.  lambda is absolute, so this
  normalisation is part of the definition (the result is not scale invariant).
* ``cg_solve`` is textbook conjugate gradient on the dense Sigma_i (reading notes
  section 2.2, Sec. 3.1: Sigma_i rho_i = mu_i solved by CG using only products
  Sigma_i p).  It exists to separate CG truncation from floating-point error;
  the reference output itself uses the exact (Cholesky) solve.
* ``lla_row_deflated_cg`` solves the same system through the exact identity
  Sigma_i = C_i + omega_i delta_i delta_i^T, with C_i the weighted key scatter about
  the weighted key mean kbar_i plus lambda I and delta_i = kbar_i - q_i (so mu_i =
  omega_i delta_i).  By Sherman-Morrison, rho_i = rho'_i / (1 + delta_i.rho'_i) with
  (C_i / omega_i) rho'_i = delta_i, the denominator is omega_i / (1 + delta_i.rho'_i),
  and b_i = sum_j wbar_ij (1 - (k_j - kbar_i).rho'_i) v_j: the softmax output minus
  a softmax-weighted value/key covariance times a probe (the form the Parallax page
  describes).  rho'_i is found by CG on the centred system; at convergence this is
  the same rho_i, but at a fixed iteration cap the iterates differ from CG on
  Sigma_i.  It is the float64 restatement of the iteration the CUDA path runs.
* ``softmax_ref`` is the Nadaraya-Watson / softmax local-constant estimate with the
  same weights (reading notes section 1, Eq. (4); kernel-methods blog chapter 1),
  the lambda -> infinity limit stated in section 2.1 (Sec. 2.3 of the paper).
* ``parallax_row`` / ``parallax_ref`` is the Parallax page's form with a caller-supplied
  probe rho (the page's learned projection W_R is trained weights, out of scope): the
  softmax output minus the softmax-weighted value/key covariance times the probe,
      out_i = sum_j wbar_ij v_j - Sigma_KV,i rho_i,
      Sigma_KV,i = sum_j wbar_ij (v_j - vbar_i)(k_j - kbar_i)^T,
  with wbar the same max-subtracted causal softmax weights normalised to sum 1, vbar_i
  and kbar_i their weighted means, and the page's boundary factor eta dropped (the page
  removes it).  The covariance matrix is formed explicitly (d x d per query).
* ``lla_row_grad`` / ``lla_grad_ref`` give the gradient of L = sum_i g_i . out_i with respect to
  q, k and v.  The pages give no backward formulas (the reading notes only say that it needs
  further linear systems, appendix D); they are derived here by differentiating Eqs. (6)-(8)
  through the exact solve: with h_j = g.v_j, den = omega - mu.rho and a_j = w_j (1 - z_j.rho),
      dL/dv_j = (a_j / den) g,   dL/dden = -(g.out)/den,
      G = -(1/den) sum_j w_j h_j z_j + (g.out/den) mu,   Sigma u = G   (the adjoint solve),
      dL/domega = dL/dden,   dL/dmu = u - rho dL/dden,   dL/dSigma = -u rho^T,
      dL/dw_j = (h_j/den)(1 - z_j.rho) + dL/domega + z_j.dL/dmu - (z_j.u)(z_j.rho),
      dL/dz_j = -(w_j h_j/den) rho + w_j dL/dmu - w_j (u (rho.z_j) + rho (u.z_j)),
  then through z_j = k_j - q_i, w_j = exp(s_j - m), s_j = tau q_i.k_j and the row maximum m
  (lambda is absolute, so the output depends on m; its gradient goes to the first index that
  attains the maximum).  ``tests/test_oracle.py`` checks it against central finite differences
  of ``lla_ref``.
* ``brute_force_fit`` minimises the weighted ridge objective of section 2.1 over
  (b, W) directly by SVD least squares, without the closed form.  Reading: the
  ridge term that reproduces Eq. (7)'s "+ lambda I" is (lambda/2)||W||_F^2 (the
  printed objective's lambda||W||_F^2 would give 2 lambda I).

Inputs are numpy arrays shaped [B, H, n, d]; whatever dtype they arrive in is
converted exactly to float64 (bf16 and fp32 values are exact in float64).
"""

from __future__ import annotations

import numpy as np
import scipy.linalg

__all__ = [
    "row_weights",
    "row_moments",
    "row_moments_split",
    "lla_row",
    "lla_ref",
    "lla_row_deflated_cg",
    "cg_centred_rounded",
    "softmax_row",
    "softmax_ref",
    "parallax_row",
    "parallax_ref",
    "lla_row_grad",
    "lla_row_grad_cg",
    "lla_grad_ref",
    "cg_solve",
    "lla_row_cg",
    "brute_force_fit",
    "ridge_objective",
    "slope_hat",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def row_weights(q_i, K_prefix, tau):
    """Max-subtracted dot-product exponential weights of one query.

    Returns (w, m) with w_j = exp(tau q_i.k_j - m), m = max_j tau q_i.k_j, over the
    causal prefix K_prefix = [k_0 .. k_i] (reading notes section 2.1 / 2.2).
    """
    q_i = _f64(q_i)
    K = _f64(K_prefix)
    logits = tau * (K @ q_i)
    m = logits.max()
    return np.exp(logits - m), m


def row_moments(q_i, K_prefix, w, lam):
    """omega, mu, Sigma of Eq. (7) from the explicit differences z_j = k_j - q_i."""
    q_i = _f64(q_i)
    Z = _f64(K_prefix) - q_i[None, :]
    omega = w.sum()
    mu = Z.T @ w
    Sigma = (Z * w[:, None]).T @ Z + lam * np.eye(q_i.shape[0])
    return omega, mu, Sigma, Z


def row_moments_split(q_i, K_prefix, w, lam):
    """The same moments through the key/query split of Eqs. (10)-(12).

    mu~ = sum_j w_j k_j, mu = mu~ - omega q;  Sigma~ = sum_j w_j k_j k_j^T + lambda I,
    Sigma = Sigma~ - mu~ q^T - q mu~^T + omega q q^T  (reading notes section 2.2).
    """
    q_i = _f64(q_i)
    K = _f64(K_prefix)
    omega = w.sum()
    mu_t = K.T @ w
    mu = mu_t - omega * q_i
    Sigma_t = (K * w[:, None]).T @ K + lam * np.eye(q_i.shape[0])
    Sigma = Sigma_t - np.outer(mu_t, q_i) - np.outer(q_i, mu_t) + omega * np.outer(q_i, q_i)
    return omega, mu_t, mu, Sigma


def _output_from_rho(w, Z, V, omega, mu, rho):
    """Eq. (8): s_j = w_j (1 - z_j.rho) / (omega - mu.rho), b = sum_j s_j v_j."""
    denom = omega - mu @ rho
    s = w * (1.0 - Z @ rho) / denom
    return s @ _f64(V), s, denom


def lla_row(q_i, K_prefix, V_prefix, tau, lam):
    """LLA output of one query from its causal prefix, exact solve (Cholesky).

    Returns a dict with out, rho, denom, omega, mu, m, s (the mixing weights s_ij)
    and cond (2-norm condition number of Sigma_i).
    """
    w, m = row_weights(q_i, K_prefix, tau)
    omega, mu, Sigma, Z = row_moments(q_i, K_prefix, w, lam)
    rho = scipy.linalg.cho_solve(scipy.linalg.cho_factor(Sigma, lower=True), mu)
    out, s, denom = _output_from_rho(w, Z, V_prefix, omega, mu, rho)
    return {"out": out, "rho": rho, "denom": denom, "omega": omega, "mu": mu,
            "m": m, "w": w, "s": s, "Sigma": Sigma}


def cg_solve(Sigma, mu, max_iters, tol):
    """Unpreconditioned conjugate gradient for Sigma x = mu, x_0 = 0.

    Rules (the pages say only "CG"; this is the reading the GPU path follows):
    the residual is kept by recurrence; before every iteration the run stops if
    ||r||_2 <= tol * ||mu||_2 (tol = 0 therefore runs exactly max_iters
    iterations unless the residual is exactly zero); mu = 0 gives x = 0 after 0
    iterations; a direction with no positive curvature (p.Sigma p <= 0, which for
    an SPD matrix means the direction has underflowed to nothing) ends the run
    without being counted.  Returns (x, iterations executed).
    """
    Sigma = _f64(Sigma)
    mu = _f64(mu)
    x = np.zeros_like(mu)
    r = mu.copy()
    p = r.copy()
    gamma = r @ r
    mu_norm = np.sqrt(gamma)
    it = 0
    while it < max_iters:
        if gamma == 0.0 or np.sqrt(gamma) <= tol * mu_norm:
            break
        Sp = Sigma @ p
        pSp = p @ Sp
        if not pSp > 0.0:
            break
        alpha = gamma / pSp
        x = x + alpha * p
        r = r - alpha * Sp
        gamma_new = r @ r
        p = r + (gamma_new / gamma) * p
        gamma = gamma_new
        it += 1
    return x, it


def lla_row_cg(q_i, K_prefix, V_prefix, tau, lam, max_iters, tol):
    """As ``lla_row`` but rho from ``cg_solve`` (truncation diagnostics)."""
    w, m = row_weights(q_i, K_prefix, tau)
    omega, mu, Sigma, Z = row_moments(q_i, K_prefix, w, lam)
    rho, iters = cg_solve(Sigma, mu, max_iters, tol)
    out, s, denom = _output_from_rho(w, Z, V_prefix, omega, mu, rho)
    return {"out": out, "rho": rho, "denom": denom, "iters": iters, "m": m, "omega": omega}


def cg_centred_rounded(Kc, wbar, lam_n, delta, max_iters, tol, u, rng):
    """``cg_solve`` on Cn = sum_j wbar_j c_j c_j^T + lam_n I (rows c_j of Kc), matrix-free, with
    every matrix-vector product perturbed the way a kernel's rounding of its product operands
    perturbs it: each coordinate of the direction p and each per-pair coefficient wbar_j (c_j.p)
    is multiplied by its own fresh factor (1 + xi), xi uniform in [-u, u], in every iteration.
    u = 0 is the unperturbed iteration.  TEST INFRASTRUCTURE: a model of rounding used only to
    measure how sensitive a capped CG result is to the arithmetic that computes it; the same
    stopping rules as ``cg_solve``.  Returns (x, iterations executed)."""
    Kc = _f64(Kc)
    wbar = _f64(wbar)
    b = _f64(delta)
    x = np.zeros_like(b)
    r = b.copy()
    p = r.copy()
    gamma = r @ r
    b_norm = np.sqrt(gamma)
    it = 0
    while it < max_iters:
        if gamma == 0.0 or np.sqrt(gamma) <= tol * b_norm:
            break
        ph = p * (1.0 + rng.uniform(-u, u, p.shape)) if u else p
        coef = wbar * (Kc @ ph)
        if u:
            coef = coef * (1.0 + rng.uniform(-u, u, coef.shape))
        Sp = Kc.T @ coef + lam_n * ph
        pSp = ph @ Sp
        if not pSp > 0.0:
            break
        alpha = gamma / pSp
        x = x + alpha * ph
        r = r - alpha * Sp
        gamma_new = r @ r
        p = r + (gamma_new / gamma) * ph
        gamma = gamma_new
        it += 1
    return x, it


def lla_row_deflated_cg(q_i, K_prefix, V_prefix, tau, lam, max_iters, tol, rounding=None):
    """LLA of one query with rho from CG on the centred key scatter.

    rounding: None (the plain float64 iteration), or (u, rng) to run the iteration through
    ``cg_centred_rounded`` with relative perturbations of size u in every product (used only to
    measure how sensitive a row's capped result is to rounding in the arithmetic).

    Steps: weights; omega, kbar = sum_j w_j k_j / omega; delta = kbar - q;
    Cn = sum_j wbar_j (k_j - kbar)(k_j - kbar)^T + (lambda/omega) I (dense);
    rho' = ``cg_solve``(Cn, delta, max_iters, tol); then
    g = 1 + delta.rho', rho = rho'/g, denom = omega/g and
    out = sum_j wbar_j (1 - (k_j - kbar).rho') v_j.
    """
    q_i = _f64(q_i)
    K = _f64(K_prefix)
    w, m = row_weights(q_i, K, tau)
    omega = w.sum()
    wbar = w / omega
    kbar = wbar @ K
    delta = kbar - q_i
    Kc = K - kbar[None, :]
    if rounding is None:
        Cn = (Kc * wbar[:, None]).T @ Kc + (lam / omega) * np.eye(q_i.shape[0])
        rho_p, iters = cg_solve(Cn, delta, max_iters, tol)
    else:
        rho_p, iters = cg_centred_rounded(Kc, wbar, lam / omega, delta, max_iters, tol, rounding[0], rounding[1])
    g = 1.0 + delta @ rho_p
    s = wbar * (1.0 - Kc @ rho_p)
    return {"out": s @ _f64(V_prefix), "rho": rho_p / g, "denom": omega / g,
            "rho_probe": rho_p, "iters": iters, "m": m, "omega": omega, "s": s}


def softmax_row(q_i, K_prefix, V_prefix, tau):
    """Local-constant (Nadaraya-Watson / softmax) estimate: sum_j (w_j/omega) v_j."""
    w, _ = row_weights(q_i, K_prefix, tau)
    return (w / w.sum()) @ _f64(V_prefix)


def _rows_iter(shape, rows):
    B, H, n, _ = shape
    if rows is None:
        for b in range(B):
            for h in range(H):
                for i in range(n):
                    yield b, h, i
    else:
        for r in rows:
            yield tuple(int(t) for t in r)


def lla_ref(q, k, v, tau, lam, rows=None, cg=None, deflated=None, rounding_u=None, rounding_seed=0):
    """Causal LLA over [B, H, n, d] inputs, row by row.

    rows: None (every (b, h, i)) or an iterable of (b, h, i) triples.
    cg: None for the exact solve, else (max_iters, tol) to solve with ``cg_solve``
        on Sigma_i; deflated: (max_iters, tol) to use ``lla_row_deflated_cg``;
    rounding_u: with ``deflated``, run its CG through ``cg_centred_rounded`` with relative
        perturbations of size rounding_u, seeded per row from (rounding_seed, b, h, i)
        (sensitivity analysis).
    Returns (out [R, d], rho [R, d], denom [R]) in float64, R rows in the order
    given (row-major over b, h, i when rows is None).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    outs, rhos, dens = [], [], []
    for b, h, i in _rows_iter(q.shape, rows):
        if deflated is not None:
            rounding = None
            if rounding_u:
                rounding = (rounding_u, np.random.Generator(np.random.PCG64([rounding_seed, b, h, i])))
            r = lla_row_deflated_cg(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], tau, lam,
                                    deflated[0], deflated[1], rounding=rounding)
        elif cg is None:
            r = lla_row(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], tau, lam)
        else:
            r = lla_row_cg(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], tau, lam, cg[0], cg[1])
        outs.append(r["out"])
        rhos.append(r["rho"])
        dens.append(r["denom"])
    d = q.shape[-1]
    return (np.array(outs).reshape(-1, d), np.array(rhos).reshape(-1, d), np.array(dens))


def softmax_ref(q, k, v, tau, rows=None):
    """Causal softmax attention with the same max-subtracted weights, row by row."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    outs = [softmax_row(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], tau)
            for b, h, i in _rows_iter(q.shape, rows)]
    return np.array(outs).reshape(-1, q.shape[-1])


def parallax_row(q_i, K_prefix, V_prefix, rho_i, tau):
    """Parallax form of one query: softmax output minus Sigma_KV rho (explicit covariance).

    Returns a dict with out, softmax (the softmax output), cov (Sigma_KV, [d_v, d_k]),
    kbar and vbar.
    """
    w, _ = row_weights(q_i, K_prefix, tau)
    wbar = w / w.sum()
    K, V = _f64(K_prefix), _f64(V_prefix)
    kbar, vbar = wbar @ K, wbar @ V
    cov = ((V - vbar[None, :]) * wbar[:, None]).T @ (K - kbar[None, :])
    soft = wbar @ V
    return {"out": soft - cov @ _f64(rho_i), "softmax": soft, "cov": cov, "kbar": kbar, "vbar": vbar}


def parallax_ref(q, k, v, rho, tau, rows=None):
    """Causal Parallax-form attention over [B, H, n, d] inputs with probe rho [B, H, n, d]."""
    q, k, v, rho = _f64(q), _f64(k), _f64(v), _f64(rho)
    outs = [parallax_row(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], rho[b, h, i], tau)["out"]
            for b, h, i in _rows_iter(q.shape, rows)]
    return np.array(outs).reshape(-1, q.shape[-1])


def lla_row_grad(q_i, K_prefix, V_prefix, g_i, tau, lam, jm=None):
    """Gradient of g_i . out_i for one query with respect to q_i, the prefix keys and values.

    Returns (out, dq [d], dK [i+1, d], dV [i+1, d]); the exact (Cholesky) solves throughout.
    jm: the key index whose logit is taken as the row maximum m (default: the first index
    attaining it).  Where two logits tie the max-subtracted definition has one-sided
    derivatives; passing the other index gives the other side.
    """
    q_i, K, V, g = _f64(q_i), _f64(K_prefix), _f64(V_prefix), _f64(g_i)
    s = tau * (K @ q_i)
    if jm is None:
        jm = int(np.argmax(s))                   # first index attaining the maximum
    w = np.exp(s - s[jm])
    omega, mu, Sigma, Z = row_moments(q_i, K, w, lam)
    fac = scipy.linalg.cho_factor(Sigma, lower=True)
    rho = scipy.linalg.cho_solve(fac, mu)
    out, s_mix, den = _output_from_rho(w, Z, V, omega, mu, rho)
    h = V @ g
    d_den = -(g @ out) / den
    G = -((w * h) @ Z) / den + (g @ out / den) * mu
    u = scipy.linalg.cho_solve(fac, G)
    d_mu = u - rho * d_den
    zr, zu = Z @ rho, Z @ u
    d_w = (h / den) * (1.0 - zr) + d_den + Z @ d_mu - zu * zr
    d_Z = (-(w * h / den))[:, None] * rho[None, :] + w[:, None] * d_mu[None, :] \
        - w[:, None] * (np.outer(zr, u) + np.outer(zu, rho))
    ds = w * d_w
    ds[jm] -= ds.sum()                           # through m = s_jm
    dq = tau * (ds @ K) - d_Z.sum(axis=0)
    dK = tau * np.outer(ds, q_i) + d_Z
    dV = np.outer(s_mix, g)
    return out, dq, dK, dV


def lla_row_grad_cg(q_i, K_prefix, V_prefix, g_i, tau, lam, max_iters, tol, jm=None):
    """The backward at a CG iteration cap: what a solver that stops early computes.

    Centred form.  With c_j = k_j - kbar, wbar_j = w_j/omega, the centred Cn and delta of
    ``lla_row_deflated_cg``, h_j = g.v_j, hbar = sum_j wbar_j h_j and tbar = sum_j wbar_j h_j c_j:
        rho' = ``cg_solve``(Cn, delta),   y = ``cg_solve``(Cn, tbar),
        Ahat_j = 1 - c_j.rho',   Bhat_j = (h_j - hbar) - c_j.y,   ds_j = wbar_j Ahat_j Bhat_j,
        sd = -(lambda/omega) rho'.y                      (the path through the row maximum)
        dv_j = wbar_j Ahat_j g,
        dk_j = tau ds_j q - wbar_j (Ahat_j y + Bhat_j rho'),   dk_jm -= tau sd q,
        dq = tau (sum_j ds_j k_j - sd k_jm) + y.
    With both solves exact this is ``lla_row_grad``: writing z_j = c_j + delta, kappa = delta.rho',
    rho = rho'/(1 + kappa), denom = omega/(1 + kappa), the exact gradient has
    1 - z_j.rho = Ahat_j/(1 + kappa), adjoint solution u = -(1 + kappa) y/omega, and the identity
    delta.y = rho'.tbar (both equal delta^T Cn^{-1} tbar) removes every term in delta.y; the sum
    of ds_j over j reduces to sd.  Returns (dq [d], dK [i+1, d], dV [i+1, d]).
    """
    q_i, K, V, g = _f64(q_i), _f64(K_prefix), _f64(V_prefix), _f64(g_i)
    s = tau * (K @ q_i)
    if jm is None:
        jm = int(np.argmax(s))
    w = np.exp(s - s[jm])
    omega = w.sum()
    wbar = w / omega
    kbar = wbar @ K
    delta = kbar - q_i
    Kc = K - kbar[None, :]
    Cn = (Kc * wbar[:, None]).T @ Kc + (lam / omega) * np.eye(q_i.shape[0])
    rho_p, _ = cg_solve(Cn, delta, max_iters, tol)
    h = V @ g
    hbar = wbar @ h
    tbar = (wbar * h) @ Kc
    y, _ = cg_solve(Cn, tbar, max_iters, tol)
    Ahat = 1.0 - Kc @ rho_p
    Bhat = (h - hbar) - Kc @ y
    ds = wbar * Ahat * Bhat
    sd = -(lam / omega) * (rho_p @ y)
    dq = tau * (ds @ K - sd * K[jm]) + y
    dK = tau * np.outer(ds, q_i) - wbar[:, None] * (Ahat[:, None] * y[None, :] + Bhat[:, None] * rho_p[None, :])
    dK[jm] -= tau * sd * q_i
    dV = np.outer(wbar * Ahat, g)
    return dq, dK, dV


def lla_grad_ref(q, k, v, dout, tau, lam, cg=None):
    """Gradients of sum_{b,h,i} dout[b,h,i] . out[b,h,i] over [B, H, n, d] inputs (float64).

    cg: None for the exact gradient (``lla_row_grad``), else (max_iters, tol) for
    ``lla_row_grad_cg``.  Returns (dq, dk, dv), each [B, H, n, d]; dk and dv sum every causal
    row's contribution.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    B, H, n, _ = q.shape
    for b in range(B):
        for h in range(H):
            for i in range(n):
                args = (q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], g[b, h, i], tau, lam)
                if cg is None:
                    _, gq, gK, gV = lla_row_grad(*args)
                else:
                    gq, gK, gV = lla_row_grad_cg(*args, cg[0], cg[1])
                dq[b, h, i] += gq
                dk[b, h, : i + 1] += gK
                dv[b, h, : i + 1] += gV
    return dq, dk, dv


def ridge_objective(b, W, q_i, K_prefix, V_prefix, w, ridge):
    """0.5 sum_j w_j ||v_j - b - W z_j||^2 + ridge ||W||_F^2 (section 2.1 objective)."""
    Z = _f64(K_prefix) - _f64(q_i)[None, :]
    R = _f64(V_prefix) - b[None, :] - Z @ W.T
    return 0.5 * np.sum(w * np.sum(R * R, axis=1)) + ridge * np.sum(W * W)


def brute_force_fit(q_i, K_prefix, V_prefix, w, ridge):
    """Minimise ``ridge_objective`` over (b, W) by SVD least squares.

    Each output coordinate is an independent weighted ridge regression on the
    augmented design [1, z_j^T]; the ridge penalty becomes d extra rows
    sqrt(2 ridge) [0, e_k^T] -> 0.  No normal equations, no closed form.
    Returns (b [d], W [d, d]).
    """
    Z = _f64(K_prefix) - _f64(q_i)[None, :]
    n, d = Z.shape
    sw = np.sqrt(_f64(w))
    A_data = sw[:, None] * np.hstack([np.ones((n, 1)), Z])
    A_ridge = np.hstack([np.zeros((d, 1)), np.sqrt(2.0 * ridge) * np.eye(d)])
    A = np.vstack([A_data, A_ridge])
    Y = np.vstack([sw[:, None] * _f64(V_prefix), np.zeros((d, _f64(V_prefix).shape[1]))])
    theta, *_ = np.linalg.lstsq(A, Y, rcond=None)
    return theta[0], theta[1:].T


def slope_hat(q_i, K_prefix, V_prefix, w, lam, b):
    """Local slope W_i of the fit, from the W normal equation at the optimum.

    With the "+ lambda I" reading: (sum_j w_j (v_j - b) z_j^T) Sigma_i^{-1}.
    Used to check Eq. (9): b_i = W_i q_i + sum_j wbar_j (v_j - W_i k_j).
    """
    omega, mu, Sigma, Z = row_moments(q_i, K_prefix, w, lam)
    C = ((_f64(V_prefix) - b[None, :]) * w[:, None]).T @ Z
    return np.linalg.solve(Sigma.T, C.T).T
