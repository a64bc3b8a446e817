"""GPU parity of the fp32 CUDA-core path against the float64 oracle.

Gates (tolerances stated here, applied per compared row):
* fp32 inputs, CG to relative residual 1e-7: out, rho and denom within 1e-4 of the exact
  (Cholesky) solve on every compared row.
* bf16 inputs (``parity_util.bf16_gate``), on every compared row, element by element: within
  (2e-2 + 3 spread) RMS(v) of the oracle's float64 centred CG at the same cap and tolerance,
  spread being that result's rounding spread at fp32's unit roundoff (2^-24), and within 2e-2
  RMS(v) of the exact solve where float64 CG has converged; finite, denom > 0.
"""
import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import workload

from parity_util import all_rows, bf16_gate, errors, oracle_rows, pick, rows_for, run_gpu, softmax_rows

pytestmark = pytest.mark.gpu
FP32 = lla.LLA_PATH_FP32


def _check_fp32(w, rows, path=FP32, gate=1e-4):
    qkv, (out, rho, den, its) = run_gpu(w, path)
    exact, _, rms_v = oracle_rows(qkv, w, rows)
    e_out, e_rho, e_den = errors(pick(out, rows), pick(rho, rows), pick(den, rows), exact, rms_v)
    assert e_out.max() <= gate, f"out err {e_out.max():.3e} at row {rows[int(e_out.argmax())]}"
    assert e_rho.max() <= gate, f"rho err {e_rho.max():.3e} at row {rows[int(e_rho.argmax())]}"
    assert e_den.max() <= gate, f"denom err {e_den.max():.3e} at row {rows[int(e_den.argmax())]}"
    assert (its.numpy() <= w.cg_max_iters).all()
    return e_out, its


def test_tiny_fp32_every_row(lla_gpu):
    w = workload("tiny_fp32")
    _check_fp32(w, all_rows(w))
    _check_fp32(w, all_rows(w), path=lla.LLA_PATH_AUTO)


def test_piecewise_fp32_ragged_small_every_row(lla_gpu):
    w = workload("piecewise_fp32", B=2, n=301)
    _check_fp32(w, all_rows(w))


@pytest.mark.slow
def test_piecewise_fp32_full_size_sampled(lla_gpu):
    w = workload("piecewise_fp32")
    _check_fp32(w, rows_for(w, 400))


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("n", [1, 31, 33, 97])
def test_fp32_path_edges_converged(lla_gpu, d, n):
    """Tiny and ragged n (one tile, tile +- 1), every d, CG run to convergence."""
    w = workload("lm_bf16", B=1, H=3, n=n, d=d, dtype="fp32", tau=1.0 / np.sqrt(d), cg_max_iters=4 * d + 64,
                 cg_tol=1e-6)
    _check_fp32(w, all_rows(w), gate=2e-4)


_bf16_gate = bf16_gate


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_fp32_path_bf16_inputs_ragged(lla_gpu, d):
    """Several query tiles and a ragged tail; 48 CG iterations so most rows converge
    (at 16 iterations nearly every row of a 333-long d=128 sequence is in the band
    where truncation dominates)."""
    w = workload("lm_bf16", B=2, H=2, n=333, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=48)
    _bf16_gate(w, all_rows(w), FP32)


@pytest.mark.slow
def test_lm_bf16_full_size_fp32_path(lla_gpu):
    w = workload("lm_bf16")
    r = _bf16_gate(w, rows_for(w, 256), FP32)
    assert (r["its"].numpy() == w.cg_max_iters).mean() > 0.99


@pytest.mark.slow
def test_long_bf16_full_size_fp32_path(lla_gpu):
    w = workload("long_bf16")
    _bf16_gate(w, rows_for(w, 64), FP32)


@pytest.mark.slow
@pytest.mark.parametrize("lam", [1e-3, 1e-1])
def test_illcond_bf16_fp32_path(lla_gpu, lam):
    w = workload("illcond_bf16", lam=lam)
    its = _bf16_gate(w, rows_for(w, 192), FP32, lam=lam)["its"]
    hist = np.bincount(its.numpy().ravel(), minlength=w.cg_max_iters + 1)
    assert hist.sum() == w.B * w.H * w.n and its.numpy().max() <= w.cg_max_iters


@pytest.mark.slow
def test_illcond_bf16_lambda_1e6_is_softmax(lla_gpu):
    w = workload("illcond_bf16", lam=1e6)
    rows = rows_for(w, 192)
    qkv, (out, rho, den, its) = run_gpu(w, FP32, lam=1e6)
    sm = softmax_rows(qkv, w, rows)
    rms_v = float(torch.sqrt(torch.mean(qkv[2].float() ** 2)))
    err = np.abs(pick(out, rows) - sm).max() / rms_v
    assert err <= 2e-2, err
