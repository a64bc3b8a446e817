"""Backward pass (lla_backward) through the C ABI against the float64 oracle.

Error metric, per gradient tensor: max over the compared entries of |gpu - ref| divided by the
RMS of ref over those entries, floored at 1e-2 RMS(dout) (the gradients are linear in dout; a
one-key prefix has dq = dk = 0 exactly, since the output is v_0 whatever q and k are).  Gates:
* adjoint CG run to convergence (relative residual 1e-6, cap 4d + 64), rho/denom from the
  oracle's exact solve (fp32): every entry of dq, dk and dv within 4e-4 of the exact gradient.
  The arithmetic is fp32 throughout, as in the fp32 forward path, which meets 2e-4 on out and
  rho under the same convergence rule.  dv_j = sum_i s_ij g_i sums the forward's per-pair
  coefficients s_ij = wbar_ij (1 - c_ij.rho'_i) down a key column instead of along a query row,
  and rho' = rho omega/denom is formed from fp32 inputs, hence twice that bound.
* the chain: the GPU forward (fp32 path, converged) feeding the GPU backward: within 1e-3 (two
  fp32 solves in series).
* at a fixed cap T (tol 0) the reference is the oracle's iteration-capped backward (CG for rho'
  and for the adjoint, T iterations each in float64): within 2e-3, the forward's fixed-cap
  bound on out.  Truncation is part of the definition being compared there.
A row whose two largest logits lie within 1e-5 relative of each other is a tie at fp32
resolution: both one-sided oracle gradients are formed and the GPU must match one of them.

Both paths are held to the same gates.  The tensor path runs the stats stage (moments, adjoint
right-hand side, adjoint CG) on tcgen05 with fp16 operands whose every rounded quantity (weights,
per-pair coefficients, CG direction) is carried as an fp16 hi + lo pair, about 22 bits, so its
error budget is that of fp32 arithmetic; q, k, v and dout are bf16 and exact in fp16.
"""
import math

import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_cotangent, make_inputs, workload
from oracle.lla_ref import lla_ref, lla_row_deflated_cg, lla_row_grad, lla_row_grad_cg

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _row_grad(qi, K, V, gi, tau, lam, cg, jm=None):
    if cg is None:
        _, dq, dK, dV = lla_row_grad(qi, K, V, gi, tau, lam, jm=jm)
        return dq, dK, dV
    return lla_row_grad_cg(qi, K, V, gi, tau, lam, cg[0], cg[1], jm=jm)


def _tie_alternative(qi, K, tau):
    """Second index of a near-tie for the maximum (None if the maximum is clear)."""
    s = tau * (K @ qi)
    if s.size < 2:
        return None
    order = np.argsort(-s, kind="stable")
    top, nxt = s[order[0]], s[order[1]]
    if top - nxt <= 1e-5 * max(1.0, abs(top)):
        first = int(np.argmax(s))
        return int(order[1]) if int(order[0]) == first else int(order[0])
    return None


def oracle_grads(qkvg, tau, lam, heads, rows_from=0, cg=None, gpu_dq=None):
    """Oracle gradients of the given (b, h) heads for query rows i >= rows_from (every key
    j >= rows_from then receives its complete dk/dv).  Near-tie rows take the one-sided
    gradient whose dq is closer to gpu_dq."""
    q, k, v, g = (t.double().numpy() for t in qkvg)
    n, d = q.shape[2], q.shape[3]
    out = {}
    for b, h in heads:
        dq = np.zeros((n, d))
        dk = np.zeros((n, d))
        dv = np.zeros((n, d))
        for i in range(rows_from, n):
            args = (q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], g[b, h, i], tau, lam, cg)
            gq, gK, gV = _row_grad(*args)
            alt = _tie_alternative(q[b, h, i], k[b, h, : i + 1], tau)
            if alt is not None and gpu_dq is not None:
                aq, aK, aV = _row_grad(*args, jm=alt)
                if np.abs(aq - gpu_dq[b, h, i]).max() < np.abs(gq - gpu_dq[b, h, i]).max():
                    gq, gK, gV = aq, aK, aV
            dq[i] = gq
            dk[: i + 1] += gK
            dv[: i + 1] += gV
        out[(b, h)] = (dq, dk, dv)
    return out


def _rel_err(gpu, ref, floor):
    scale = max(math.sqrt(float(np.mean(ref ** 2))), floor)
    return float(np.abs(gpu - ref).max()) / scale


def _run_backward(w, qkvg, rho, den, T, tol, return_iters=True, path=lla.LLA_PATH_FP32):
    q, k, v, g = (t.to(DEV) for t in qkvg)
    res = lla.backward(q, k, v, rho.to(DEV), den.to(DEV), g, w.tau, w.lam, T, tol, path=path,
                       return_iters=return_iters)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return [t.cpu() for t in res]


def _exact_rho(qkv, w):
    qn, kn, vn = (t.double().numpy() for t in qkv)
    _, rho, den = lla_ref(qn, kn, vn, w.tau, w.lam)
    shape = (w.B, w.H, w.n)
    return (torch.from_numpy(rho.reshape(*shape, w.d)).float(), torch.from_numpy(den.reshape(shape)).float())


def _compare(w, qkvg, grads, gate, heads=None, rows_from=0, cg=None):
    dq, dk, dv = (t.double().numpy() for t in grads[:3])
    heads = [(b, h) for b in range(w.B) for h in range(w.H)] if heads is None else heads
    ref = oracle_grads(qkvg, w.tau, w.lam, heads, rows_from, cg, gpu_dq=dq)
    sl = slice(rows_from, None)
    floor = 1e-2 * math.sqrt(float(np.mean(qkvg[3].double().numpy() ** 2)))
    for name, gpu, idx in (("dq", dq, 0), ("dk", dk, 1), ("dv", dv, 2)):
        a = np.stack([gpu[b, h, sl] for b, h in heads])
        r = np.stack([ref[bh][idx][sl] for bh in heads])
        assert np.isfinite(a).all(), f"{name} not finite"
        e = _rel_err(a, r, floor)
        assert e <= gate, f"{name} err {e:.3e} RMS"
    return ref


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("n", [1, 31, 33, 97])
def test_backward_converged_every_entry(lla_gpu, d, n):
    """One tile, tile +- 1 and a ragged multi-tile tail, every head dim; fp32 inputs."""
    w = workload("lm_bf16", B=1, H=2, n=n, d=d, dtype="fp32", tau=1.0 / np.sqrt(d))
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    grads = _run_backward(w, (*qkv, g), rho, den, 4 * d + 64, 1e-6)
    assert (grads[3].numpy() <= 4 * d + 64).all()
    _compare(w, (*qkv, g), grads, 4e-4)


PATHS = [pytest.param(lla.LLA_PATH_FP32, id="fp32"), pytest.param(lla.LLA_PATH_TENSOR, id="tensor")]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d", [64, 128])
def test_backward_bf16_inputs_ragged(lla_gpu, d, path):
    """bf16 q, k, v and dout (exact in float64 too), several query tiles and a ragged tail."""
    w = workload("lm_bf16", B=2, H=2, n=333, d=d, tau=1.0 / np.sqrt(d))
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    grads = _run_backward(w, (*qkv, g), rho, den, 4 * d + 64, 1e-6, path=path)
    _compare(w, (*qkv, g), grads, 4e-4)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 257])
def test_backward_tensor_path_edges(lla_gpu, d, n):
    """The tensor path at tile boundaries and on rank-deficient short prefixes (n < d)."""
    w = workload("lm_bf16", B=1, H=2, n=n, d=d, tau=1.0 / np.sqrt(d))
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    grads = _run_backward(w, (*qkv, g), rho, den, 4 * d + 64, 1e-6, path=lla.LLA_PATH_TENSOR)
    _compare(w, (*qkv, g), grads, 4e-4)


def test_backward_small_lambda_piecewise(lla_gpu):
    """The piecewise-linear workload (lambda 1e-2, tau 4): ill-conditioned early rows."""
    w = workload("piecewise_fp32", B=1, H=2, n=161)
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    grads = _run_backward(w, (*qkv, g), rho, den, 4 * w.d + 64, 1e-6)
    _compare(w, (*qkv, g), grads, 4e-4)


def test_backward_after_gpu_forward(lla_gpu):
    """The chain a training step runs: GPU forward (fp32 path, converged), then the backward."""
    w = workload("lm_bf16", B=1, H=3, n=200, d=64, dtype="fp32", tau=0.125)
    qkv = make_inputs(w)
    g = make_cotangent(w)
    q, k, v = (t.to(DEV) for t in qkv)
    _, rho, den = lla.forward(q, k, v, w.tau, w.lam, 4 * w.d + 64, 1e-6, path=lla.LLA_PATH_FP32)
    grads = _run_backward(w, (*qkv, g), rho.cpu(), den.cpu(), 4 * w.d + 64, 1e-6)
    _compare(w, (*qkv, g), grads, 1e-3)


@pytest.mark.parametrize("path", PATHS)
def test_backward_fixed_cap_matches_capped_oracle(lla_gpu, path):
    """The LM configuration's cap T = 16 (tol 0) on a 1100-long bf16 sequence: rho/denom from the
    GPU fp32 forward at the same cap, the reference is the oracle's capped backward, compared on
    the last 64 positions (their dk/dv need only the rows after them).  Those rows see about 300
    effective keys: CG at 16 iterations is in the regime where its fp32 and float64 iterates
    agree.  On short prefixes (effective keys below d) 16 iterations leave the solve far from
    converged (the capped float64 gradient is up to 0.5 RMS away from the exact one) and the fp32
    and float64 iterates drift apart by a few percent; those rows are checked for finiteness
    here and for correctness by the converged tests above."""
    w = workload("lm_bf16", B=1, H=2, n=1100)
    qkv = make_inputs(w)
    g = make_cotangent(w)
    q, k, v = (t.to(DEV) for t in qkv)
    _, rho, den = lla.forward(q, k, v, w.tau, w.lam, w.cg_max_iters, 0.0, path=lla.LLA_PATH_FP32)
    grads = _run_backward(w, (*qkv, g), rho.cpu(), den.cpu(), w.cg_max_iters, 0.0, path=path)
    its = grads[3].numpy()
    assert (its <= w.cg_max_iters).all() and (its == w.cg_max_iters).mean() > 0.95
    for t in grads[:3]:
        assert torch.isfinite(t).all()
    _compare(w, (*qkv, g), grads, 2e-3, rows_from=w.n - 64, cg=(w.cg_max_iters, 0.0))


@pytest.mark.parametrize("path", PATHS)
def test_backward_is_deterministic_and_takes_a_workspace(lla_gpu, path):
    """No atomics on the data path: two runs agree bit for bit, with the pool's scratch or the caller's."""
    w = workload("lm_bf16", B=2, H=2, n=130, d=64, tau=0.125)
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    a = _run_backward(w, (*qkv, g), rho, den, 24, 0.0, return_iters=False, path=path)
    ws = torch.empty(lla.lla_backward_workspace_size(lla.LLA_DTYPE_BF16, path, w.B, w.H, w.n, w.d),
                     dtype=torch.uint8, device=DEV)
    q, k, v, gg = (t.to(DEV) for t in (*qkv, g))
    b = lla.backward(q, k, v, rho.to(DEV), den.to(DEV), gg, w.tau, w.lam, 24, 0.0, path=path, workspace=ws)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y.cpu())


def test_backward_single_key_rows(lla_gpu):
    """n = 1: one key, so c = k - kbar = 0, the adjoint right-hand side is 0, y = 0, and dv equals
    dout up to the rounding of 1 - c.rho' (evaluated as k.rho' - kbar.rho')."""
    w = workload("lm_bf16", B=3, H=2, n=1, d=32, dtype="fp32", tau=0.2)
    qkv = make_inputs(w)
    g = make_cotangent(w)
    rho, den = _exact_rho(qkv, w)
    grads = _run_backward(w, (*qkv, g), rho, den, 8, 0.0)
    assert torch.allclose(grads[2], g.float(), rtol=1e-4, atol=1e-6)
    _compare(w, (*qkv, g), grads, 4e-4)


@pytest.mark.slow
def test_backward_lm_full_size_sampled(lla_gpu):
    """The LM workload at full size (8 x 16 heads x 4096, d = 128, bf16) in the configuration the
    benchmark times (T = 16, tol 0, the default path: tensor stats stage): dq, dk and dv of the last 40 positions of two heads (their
    dk/dv need every later row: 40 oracle rows each) against the capped oracle; every entry of
    every head finite."""
    w = workload("lm_bf16")
    qkv = make_inputs(w)
    g = make_cotangent(w)
    q, k, v = (t.to(DEV) for t in qkv)
    _, rho, den = lla.forward(q, k, v, w.tau, w.lam, w.cg_max_iters, 0.0, path=lla.LLA_PATH_FP32)
    del q, k, v
    grads = _run_backward(w, (*qkv, g), rho.cpu(), den.cpu(), w.cg_max_iters, 0.0, return_iters=False,
                          path=lla.LLA_PATH_AUTO)
    for t in grads:
        assert torch.isfinite(t).all()
    _compare(w, (*qkv, g), grads, 2e-3, heads=[(0, 0), (w.B - 1, w.H - 1)], rows_from=w.n - 40,
             cg=(w.cg_max_iters, 0.0))
