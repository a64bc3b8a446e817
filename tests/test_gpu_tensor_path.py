"""GPU parity of the tcgen05 tensor-core path (bf16 inputs, fp16 operands, fp32 state)
against the float64 oracle.

Gate (``parity_util.bf16_gate``), on every compared row, element by element:
* against the oracle's float64 centred CG at the same cap and tolerance, within
  (2e-2 + 3 spread) RMS(v), spread being how far that capped result moves when every product is
  perturbed at the path's unit roundoff (fp16 coefficients at a fixed cap: 2^-11; the precise
  hi + lo form of tolerance mode: 2^-22).  Rows whose capped result is insensitive to rounding
  are held to 2e-2; in the band of short prefixes where truncated CG is roundoff-sensitive the
  bound widens by what the oracle measures;
* against the exact solve within 2e-2 RMS(v) on the rows where float64 CG has converged;
* finite, denom > 0.
The output is bf16, so one output ulp is already 4e-3 to 1.6e-2 RMS(v) for |out| in [0.5, 4).
"""
import math

import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload

from parity_util import (all_rows, bf16_gate, oracle_rows, path_unit_roundoff, pick, rounding_spread, rows_for,
                         run_gpu, softmax_rows)

pytestmark = pytest.mark.gpu
TC = lla.LLA_PATH_TENSOR


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 64, 127, 128, 129, 333])
def test_tensor_path_tiles_and_ragged_tails(lla_gpu, d, n):
    """One tile, tile +- 1, several tiles with a ragged tail; CG run long enough to converge, so
    every row is held to 2e-2 of the float64 CG result."""
    w = workload("lm_bf16", B=2, H=2, n=n, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=64)
    r = bf16_gate(w, all_rows(w), TC, max_loose_frac=0.01)
    assert r["stats"]["truncated_frac"] <= 0.01


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_path_ragged_at_the_lm_cap(lla_gpu, d):
    """The LM cap (16 iterations) on a ragged multi-tile shape: here most rows below ~3d are
    in the truncation band, and the bound there widens by the oracle's rounding spread."""
    w = workload("lm_bf16", B=2, H=2, n=333, d=d, tau=1.0 / np.sqrt(d))
    r = bf16_gate(w, all_rows(w), TC)
    late = r["stats"]["bands"].get("128-512")
    assert late is not None and late["rows"] > 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 129, 300])
def test_tensor_path_tolerance_mode(lla_gpu, d, n):
    """cg_tol > 0: per-query stopping (the precise hi + lo form, launched without MAX sweeps: one
    row, a tile and one, a ragged multi-tile shape); iteration counts within the cap."""
    w = workload("lm_bf16", B=1, H=3, n=n, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=96, cg_tol=1e-5)
    r = bf16_gate(w, all_rows(w), TC, max_loose_frac=0.01)
    its = r["its"].numpy()
    assert its.max() <= 96 and its.min() >= 1


def test_tensor_path_matches_fp32_path_at_fixed_cap(lla_gpu):
    """Same inputs through both GPU paths at T=16 (truncated CG), element by element on sampled
    rows: |tc - fp32| <= (2e-2 + 3 (spread_tc + spread_fp32)) RMS(v), the spreads being the
    oracle's rounding spreads at each path's unit roundoff."""
    w = workload("lm_bf16", B=2, H=4, n=1000)
    qkv, (o_tc, r_tc, d_tc, i_tc) = run_gpu(w, TC)
    _, (o_32, r_32, d_32, i_32) = run_gpu(w, lla.LLA_PATH_FP32, inputs=qkv)
    rows = rows_for(w, 400)
    _, cg, rms_v = oracle_rows(qkv, w, rows)
    sp_tc = rounding_spread(qkv, w, rows, path_unit_roundoff(w, TC, 0.0), cg[0], rms_v)
    sp_32 = rounding_spread(qkv, w, rows, path_unit_roundoff(w, lla.LLA_PATH_FP32, 0.0), cg[0], rms_v)
    diff = np.abs(pick(o_tc, rows) - pick(o_32, rows)).max(axis=1) / rms_v
    bound = 2e-2 + 3.0 * (sp_tc + sp_32)
    bad = np.nonzero(diff > bound)[0]
    assert bad.size == 0, [(rows[j], float(diff[j]), float(bound[j])) for j in bad[:6]]
    assert (d_tc > 0).all() and torch.isfinite(o_tc.float()).all()


def _wide_range_inputs(w, k_outlier):
    q, k, v = (t.clone() for t in make_inputs(w))
    v[0, 1] = (v[0, 1].float() * 1000).bfloat16()
    q[0, 2] = (q[0, 2].float() * 2.0 ** -6).bfloat16()
    k[0, 2] = (k[0, 2].float() * 2.0 ** -6).bfloat16()
    k[1, 2, 100, 5] = k_outlier
    v[1, 3, 200, 7] = -5000.0
    return q, k, v


def _wide_range_errors(w, inputs, rows):
    """Per row and element: |out - out_cg| / (2e-2 RMS(v of the row's head) + 2^-8 |out_cg|)."""
    q, k, v = inputs
    qkv, (out, rho, den, its) = run_gpu(w, TC, inputs=inputs)
    _, cg, _ = oracle_rows(qkv, w, rows)
    rms_slice = torch.sqrt((v.double() ** 2).mean(dim=(-1, -2))).numpy()
    rms_row = np.array([rms_slice[b, h] for b, h, _ in rows])[:, None]
    g = pick(out, rows)
    assert np.isfinite(g).all() and (pick(den, rows) > 0).all()
    return np.abs(g - cg[0]) / (2e-2 * rms_row + 2.0 ** -8 * np.abs(cg[0]))


def test_tensor_path_wide_dynamic_range(lla_gpu):
    """One head of v scaled by 10^3, one head of q and k by 2^-6 (their logits by 2^-12), a key
    with one coordinate at 30 (30 times the keys' RMS) and a value at -5000; CG to convergence.
    Every head keeps its precision: every row within 2e-2 of its own head's RMS(v) plus 2^-8 |out|
    (the bf16 output rounding, which dominates next to the value outlier) of the float64 CG result."""
    w = workload("lm_bf16", B=2, H=4, n=600, cg_max_iters=64)
    rows = all_rows(w)[::3]
    err = _wide_range_errors(w, _wide_range_inputs(w, 30.0), rows)
    worst = np.argsort(-err.max(axis=1))[:6]
    assert err.max() <= 1.0, [(rows[j], float(err[j].max())) for j in worst]


@pytest.mark.xfail(strict=True, reason=(
    "a key 300 times the keys' RMS: rows whose weight sits on it have |kbar| ~ 300 and rho' ~ 200, "
    "and the centred output moves by (error of kbar) . rho' times (vbar - out); kbar's fp32 rounding "
    "alone gives 1e-2 to 3e-2 (the fp32 path misses by that much too), its fp16 weights about 0.08"))
def test_tensor_path_extreme_key_outlier_is_conditioning_limited(lla_gpu):
    w = workload("lm_bf16", B=2, H=4, n=600, cg_max_iters=64)
    rows = [(1, 2, i) for i in range(90, 600, 3)]
    err = _wide_range_errors(w, _wide_range_inputs(w, 300.0), rows)
    assert err.max() <= 1.0


@pytest.mark.slow
def test_lm_bf16_full_size_tensor_path(lla_gpu):
    w = workload("lm_bf16")
    r = bf16_gate(w, rows_for(w, 256), TC)
    assert (r["its"].numpy() <= w.cg_max_iters).all()


@pytest.mark.slow
def test_long_bf16_full_size_tensor_path(lla_gpu):
    """n = 32768: also checks that the call's device footprint is Theta(n d)."""
    w = workload("long_bf16")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    bf16_gate(w, rows_for(w, 64), TC)
    peak = torch.cuda.max_memory_allocated() - base
    nd = w.B * w.H * w.n * w.d
    # q,k,v,out bf16 + rho fp32 + iters/denom + workspace (3 fp16 copies + fp32 kbar): < 40 bytes per element
    assert peak < 40 * nd, peak


@pytest.mark.slow
@pytest.mark.parametrize("lam", [1e-3, 1e-1])
def test_illcond_bf16_through_lla_forward(lla_gpu, lam):
    """The ill-conditioned workload (B=4, H=8, n=8192, d=64, CG to 1e-4, cap 64) through the C
    entry point lla_forward itself (bf16, automatic path: the tensor path's precise form)."""
    w = workload("illcond_bf16", lam=lam)
    bf16_gate(w, rows_for(w, 192), lla.LLA_PATH_AUTO, lam=lam, entry="lla_forward")
    _, (_, _, _, its) = run_gpu(w, lla.LLA_PATH_AUTO, lam=lam)
    hist = np.bincount(its.numpy().ravel(), minlength=w.cg_max_iters + 1)
    assert hist.sum() == w.B * w.H * w.n and its.numpy().max() <= w.cg_max_iters


@pytest.mark.slow
def test_illcond_bf16_lambda_1e6_is_softmax_through_lla_forward(lla_gpu):
    w = workload("illcond_bf16", lam=1e6)
    rows = rows_for(w, 192)
    qkv, (out, rho, den, its) = run_gpu(w, lla.LLA_PATH_AUTO, lam=1e6, entry="lla_forward")
    sm = softmax_rows(qkv, w, rows)
    rms_v = float(torch.sqrt(torch.mean(qkv[2].float() ** 2)))
    assert np.abs(pick(out, rows) - sm).max() / rms_v <= 2e-2


def _rows_past_first_block_headroom(q, k, tau):
    """Rows whose causal maximum of tau q.k exceeds the maximum over the first 128 keys by more than
    7.5 in log2 units: the launch without a MAX sweep cannot hold their weights in fp16 and marks
    their tiles for the second launch, which redoes them with one."""
    qd, kd = q.double(), k.double()
    s = tau * torch.einsum("bhid,bhjd->bhij", qd, kd)
    n = s.shape[-1]
    causal = torch.ones(n, n, dtype=torch.bool).tril()
    s = s.masked_fill(~causal, -math.inf)
    jump = (s.amax(-1) - s[..., :128].amax(-1)) * (1.0 / math.log(2.0))
    return int((jump > 7.5).sum())


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_path_row_maximum_far_past_the_first_block(lla_gpu, d):
    """Tolerance mode (the precise form, launched without MAX sweeps).  Keys 128..255 scaled by 4, so
    most rows past the first tile have their maximum far above the first key block's: those tiles are
    redone by the MAX-sweep launch.  Every row within 2e-2 of the float64 CG at the same tolerance."""
    w = workload("lm_bf16", B=1, H=2, n=300, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=96, cg_tol=1e-5)
    q, k, v = (t.clone() for t in make_inputs(w))
    k[:, :, 128:256] = (k[:, :, 128:256].float() * 4.0).bfloat16()
    assert _rows_past_first_block_headroom(q, k, w.tau) > 100
    bf16_gate(w, all_rows(w), TC, inputs=(q, k, v), max_loose_frac=0.01)
