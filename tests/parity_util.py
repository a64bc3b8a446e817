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


def run_gpu(w, path, lam=None, tol=None, iters=None, return_iters=True, inputs=None, entry="forward"):
    """Run the CUDA path on w's seeded inputs (or the given ones).  entry="lla_forward" calls the
    C entry point lla_forward itself (bf16, automatic path; no iteration counts: its is None)."""
    q, k, v = make_inputs(w) if inputs is None else inputs
    dev = torch.device("cuda:0")
    lam = w.lam if lam is None else lam
    iters = w.cg_max_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if entry == "lla_forward":
        out = torch.empty_like(qd)
        rho = torch.empty(qd.shape, dtype=torch.float32, device=dev)
        den = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
        lla.lla_forward(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), rho.data_ptr(), den.data_ptr(),
                        w.B, w.H, w.n, w.d, w.tau, lam, iters, tol, torch.cuda.current_stream().cuda_stream)
        res = (out, rho, den, None)
    else:
        res = lla.forward(qd, kd, vd, w.tau, lam, iters, tol, path=path, return_iters=return_iters)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    host = [t.cpu() if t is not None else None for t in res]
    return (q, k, v), host


def pick(arr, rows):
    a = arr.double().numpy() if isinstance(arr, torch.Tensor) else arr
    return np.array([a[b, h, i] for b, h, i in rows])


def oracle_rows(qkv, w, rows, lam=None, iters=None, tol=None):
    """Exact solve and the float64 centred CG at the same cap and tolerance, on the rows."""
    qn, kn, vn = (t.double().numpy() for t in qkv)
    lam = w.lam if lam is None else lam
    T = w.cg_max_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    exact = lla_ref(qn, kn, vn, w.tau, lam, rows=rows)
    cg = lla_ref(qn, kn, vn, w.tau, lam, rows=rows, deflated=(T, tol))
    rms_v = math.sqrt(float(np.mean(vn ** 2)))
    return exact, cg, rms_v


def rounding_spread(qkv, w, rows, u, cg_out, rms_v, lam=None, iters=None, tol=None, seeds=3):
    """Per row: how far the float64 centred CG result at the cap moves when every product of every
    iteration is perturbed at relative size u (``cg_centred_rounded``), max over a few seeds, in
    units of RMS(v).  Computed by the oracle alone; it measures how sensitive the capped result is
    to the arithmetic, whatever computes it."""
    qn, kn, vn = (t.double().numpy() for t in qkv)
    lam = w.lam if lam is None else lam
    T = w.cg_max_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    spread = np.zeros(len(rows))
    for seed in range(seeds):
        o = lla_ref(qn, kn, vn, w.tau, lam, rows=rows, deflated=(T, tol), rounding_u=u, rounding_seed=seed)[0]
        spread = np.maximum(spread, np.abs(o - cg_out).max(axis=1) / rms_v)
    return spread


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


# Relative error of the per-pair coefficients each GPU path forms, for the rounding model.
# * Tensor path at a fixed cap: fp16 rounding of the coefficients, 2^-11.
# * fp32 path, and the tensor path's precise (hi + lo) form: the coefficient w (k.p - kbar.p) is
#   formed from two fp32 dot products over the head dimension, so its error is a few ulps of |k||p|,
#   many ulps of the difference where it cancels.  A float32 emulation of that arithmetic on LM rows
#   measured relative errors of 2^-22.4 (median), 2^-20.3 (90%) and 2^-17 (99%); the model's uniform
#   perturbation in [-u, u] takes u = 2^-20, the 90% figure (the precise form's hi + lo split, about
#   2^-22, is below it).
def path_unit_roundoff(w, path, cg_tol):
    dtype = lla.LLA_DTYPE_BF16 if w.dtype == "bf16" else lla.LLA_DTYPE_FP32
    if lla.lla_resolve_path(dtype, path, w.d) == lla.LLA_PATH_FP32:
        return 2.0 ** -20
    return 2.0 ** -20 if cg_tol > 0 else 2.0 ** -11


POSITION_BANDS = [(0, 16), (16, 128), (128, 512), (512, 1 << 30)]


def bf16_gate(w, rows, path, lam=None, tol=None, iters=None, gate=2e-2, conv_tol=2e-3, k_spread=3.0,
              inputs=None, max_loose_frac=None, entry="forward"):
    """Run the GPU path and check out on EVERY compared row, element by element:

    (1) against the oracle's float64 centred CG at the same cap and tolerance:
            max_e |out - out_cg| <= (gate + k_spread * spread) RMS(v),
        spread being the row's rounding spread at the path's unit roundoff (``rounding_spread``).
        On rows whose capped CG result is insensitive to rounding the bound is the gate itself;
        where truncated CG is roundoff-sensitive (a band of short prefixes at a small cap, where
        even float32 arithmetic of the same steps moves the result by O(RMS(v))) it widens by
        what the oracle measures there, never more;
    (2) against the exact (Cholesky) solve at the gate, on the rows where the oracle's own
        float64 CG has converged (within conv_tol of the exact solve) and whose result is not
        roundoff-sensitive (spread <= gate / 2: a row can converge in float64 yet not in the
        path's arithmetic);
    (3) finite everywhere, denom > 0.
    max_loose_frac: if given, at most this fraction of rows may have a widened bound (spread >
    gate / 2).  Returns a dict of per-row errors, iteration counts and the fractions by band."""
    cg_tol = w.cg_tol if tol is None else tol
    qkv, (out, rho, den, its) = run_gpu(w, path, lam=lam, tol=tol, iters=iters, inputs=inputs, entry=entry)
    exact, cg, rms_v = oracle_rows(qkv, w, rows, lam=lam, iters=iters, tol=tol)
    spread = rounding_spread(qkv, w, rows, path_unit_roundoff(w, path, cg_tol), cg[0], rms_v, lam=lam, iters=iters,
                             tol=tol)
    g_out, g_rho, g_den = pick(out, rows), pick(rho, rows), pick(den, rows)
    assert np.isfinite(g_out).all() and np.isfinite(g_rho).all() and (g_den > 0).all()
    e_cg = np.abs(g_out - cg[0]).max(axis=1) / rms_v
    e_ex = np.abs(g_out - exact[0]).max(axis=1) / rms_v
    trunc = np.abs(cg[0] - exact[0]).max(axis=1) / rms_v
    bound = gate + k_spread * spread
    bad = np.nonzero(e_cg > bound)[0]
    assert bad.size == 0, (f"{bad.size} rows over the bound vs float64 CG at the cap: worst "
                           f"{[(rows[j], round(float(e_cg[j]), 4), round(float(bound[j]), 4)) for j in bad[:6]]}")
    conv = trunc <= conv_tol
    loose = spread > gate / 2
    bad = np.nonzero(conv & ~loose & (e_ex > gate))[0]
    assert bad.size == 0, (f"{bad.size} converged rows over {gate} vs the exact solve: worst "
                           f"{[(rows[j], round(float(e_ex[j]), 4)) for j in bad[:6]]}")
    pos = np.array([r[2] for r in rows])
    bands = {}
    for lo, hi in POSITION_BANDS:
        m = (pos >= lo) & (pos < hi)
        if m.any():
            bands[f"{lo}-{hi}"] = {"rows": int(m.sum()), "widened": float(loose[m].mean()),
                                   "truncated": float((~conv[m]).mean()),
                                   "max_err_vs_cg": float(e_cg[m].max()),
                                   "max_err_vs_cg_unwidened": float(e_cg[m & ~loose].max()) if (m & ~loose).any()
                                   else None}
    stats = {"rows": len(rows), "widened_frac": float(loose.mean()), "truncated_frac": float((~conv).mean()),
             "max_err_vs_cg_unwidened": float(e_cg[~loose].max()) if (~loose).any() else None,
             "max_err_vs_exact_converged": float(e_ex[conv & ~loose].max()) if (conv & ~loose).any() else None,
             "bands": bands}
    print(f"[parity] {w.name} B={w.B} H={w.H} n={w.n} d={w.d} path={path}: {stats}")
    if max_loose_frac is not None:
        assert loose.mean() <= max_loose_frac, f"{loose.mean():.3f} of rows roundoff-sensitive"
    return {"e_cg": e_cg, "e_ex": e_ex, "spread": spread, "conv": conv, "its": its, "stats": stats}
