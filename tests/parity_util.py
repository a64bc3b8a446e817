"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle on the
same inputs, and compare with the error metrics stated in the tests.

Metrics (per compared row, then the max over rows):
* out:   max_e |out - ref| / RMS(v), RMS over the whole v tensor;
* rho:   max_e |rho - ref| / RMS(ref rho over the compared rows);
* denom: |denom - ref| / ref.
"""
import math

import numpy as np
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, sample_rows
from oracle.lla_ref import lla_ref, softmax_ref


def run_gpu(w, path, lam=None, tol=None, iters=None, return_iters=True, inputs=None):
    q, k, v = make_inputs(w) if inputs is None else inputs
    dev = torch.device("cuda:0")
    res = lla.forward(q.to(dev), k.to(dev), v.to(dev), w.tau, w.lam if lam is None else lam,
                      w.cg_max_iters if iters is None else iters, w.cg_tol if tol is None else tol,
                      path=path, return_iters=return_iters)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    host = [t.cpu() for t in res]
    return (q, k, v), host


def pick(arr, rows):
    a = arr.double().numpy() if isinstance(arr, torch.Tensor) else arr
    return np.array([a[b, h, i] for b, h, i in rows])


def oracle_rows(qkv, w, rows, lam=None, iters=None, tol=None, sensitivity=False):
    """Exact solve and float64 CG (same cap/tol) on the rows; with sensitivity=True also the
    CG result with every weight perturbed by up to 2^-10 relative (fp16 coefficient resolution)."""
    qn, kn, vn = (t.double().numpy() for t in qkv)
    lam = w.lam if lam is None else lam
    T = w.cg_max_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    exact = lla_ref(qn, kn, vn, w.tau, lam, rows=rows)
    cg = lla_ref(qn, kn, vn, w.tau, lam, rows=rows, deflated=(T, tol))
    rms_v = math.sqrt(float(np.mean(vn ** 2)))
    if not sensitivity:
        return exact, cg, rms_v
    pert = lla_ref(qn, kn, vn, w.tau, lam, rows=rows, deflated=(T, tol), noise_rel=2.0 ** -10)
    return exact, cg, rms_v, pert


def errors(g_out, g_rho, g_den, ref, rms_v):
    r_out, r_rho, r_den = ref
    e_out = np.abs(g_out - r_out).max(axis=1) / rms_v
    rms_rho = math.sqrt(float(np.mean(r_rho ** 2))) or 1.0
    e_rho = np.abs(g_rho - r_rho).max(axis=1) / rms_rho
    e_den = np.abs(g_den - r_den) / np.abs(r_den)
    return e_out, e_rho, e_den


def all_rows(w):
    return [(b, h, i) for b in range(w.B) for h in range(w.H) for i in range(w.n)]


def rows_for(w, count):
    return sample_rows(w, count) if w.B * w.H * w.n > count else all_rows(w)


def softmax_rows(qkv, w, rows):
    qn, kn, vn = (t.double().numpy() for t in qkv)
    return softmax_ref(qn, kn, vn, w.tau, rows=rows)


def bf16_gate(w, rows, path, lam=None, tol=None, iters=None, gate=2e-2, min_ok_frac=0.5, conv_tol=2e-3,
              sens_tol=5e-3):
    """Run the GPU path and gate out against the exact solve on the rows that are
    (a) converged: the oracle's own float64 CG at the same cap and tolerance is within
        conv_tol RMS(v) of the exact solve, and
    (b) stable: perturbing every weight by up to 2^-10 relative (the resolution of the
        tensor path's fp16 per-pair coefficients) moves the float64 CG result by at most
        sens_tol RMS(v).
    Both criteria are computed by the oracle alone.  Every row must be finite with
    denom > 0.  Returns (per-row out error vs exact, gated mask, iteration counts)."""
    qkv, (out, rho, den, its) = run_gpu(w, path, lam=lam, tol=tol, iters=iters)
    exact, cg, rms_v, pert = oracle_rows(qkv, w, rows, lam=lam, iters=iters, tol=tol, sensitivity=True)
    g_out, g_rho, g_den = pick(out, rows), pick(rho, rows), pick(den, rows)
    assert np.isfinite(g_out).all() and np.isfinite(g_rho).all() and (g_den > 0).all()
    trunc = np.abs(cg[0] - exact[0]).max(axis=1) / rms_v
    sens = np.abs(pert[0] - cg[0]).max(axis=1) / rms_v
    ok = (trunc <= conv_tol) & (sens <= sens_tol)
    assert ok.mean() >= min_ok_frac, f"only {ok.mean():.2f} of rows converged in the oracle"
    e_out, e_rho, e_den = errors(g_out, g_rho, g_den, exact, rms_v)
    bad = np.nonzero(ok & (e_out > gate))[0]
    assert bad.size == 0, (f"{bad.size} converged rows over {gate}: worst {e_out[ok].max():.3e} "
                           f"at {rows[int(np.argmax(np.where(ok, e_out, -1)))]}")
    return e_out, ok, its
