"""GPU parity of the tcgen05 tensor-core path (bf16 inputs, fp16 operands, fp32 state)
against the float64 oracle.

Gate (as for the fp32 path on bf16 inputs): out within 2e-2 RMS(v) of the exact solve on
every compared row where the oracle's own float64 CG at the same iteration cap has
converged; all rows finite with denom > 0.  The output is bf16, so one output ulp is
already 4e-3 to 1.6e-2 RMS(v) for |out| in [0.5, 4).
"""
import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import workload

from parity_util import all_rows, bf16_gate, pick, rows_for, run_gpu, softmax_rows

pytestmark = pytest.mark.gpu
TC = lla.LLA_PATH_TENSOR


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 64, 127, 128, 129, 333])
def test_tensor_path_tiles_and_ragged_tails(lla_gpu, d, n):
    """One tile, tile +- 1, several tiles with a ragged tail; CG run long enough to converge."""
    w = workload("lm_bf16", B=2, H=2, n=n, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=64)
    bf16_gate(w, all_rows(w), TC, min_ok_frac=0.5)


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_path_tolerance_mode(lla_gpu, d):
    """cg_tol > 0: per-query stopping; iteration counts within the cap."""
    w = workload("lm_bf16", B=1, H=3, n=300, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=96, cg_tol=1e-5)
    e, ok, its = bf16_gate(w, all_rows(w), TC, min_ok_frac=0.5)
    assert its.numpy().max() <= 96 and its.numpy().min() >= 1


def test_tensor_path_matches_fp32_path_at_fixed_cap(lla_gpu):
    """Same inputs through both GPU paths at T=16 (truncated CG): medians agree at the
    bf16 output resolution; the truncation band differs (it is roundoff-sensitive)."""
    w = workload("lm_bf16", B=2, H=4, n=1000)
    qkv, (o_tc, r_tc, d_tc, i_tc) = run_gpu(w, TC)
    _, (o_32, r_32, d_32, i_32) = run_gpu(w, lla.LLA_PATH_FP32, inputs=qkv)
    rms_v = float(torch.sqrt(torch.mean(qkv[2].float() ** 2)))
    diff = (o_tc.float() - o_32.float()).abs().amax(-1) / rms_v
    assert float(diff.median()) <= 1.6e-2
    assert (d_tc > 0).all() and torch.isfinite(o_tc.float()).all()


@pytest.mark.slow
def test_lm_bf16_full_size_tensor_path(lla_gpu):
    w = workload("lm_bf16")
    e, ok, its = bf16_gate(w, rows_for(w, 256), TC)
    assert (its.numpy() <= w.cg_max_iters).all()


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
def test_illcond_bf16_lambda_1e6_is_softmax_tensor_path(lla_gpu):
    w = workload("illcond_bf16", lam=1e6)
    rows = rows_for(w, 192)
    qkv, (out, rho, den, its) = run_gpu(w, TC, lam=1e6)
    sm = softmax_rows(qkv, w, rows)
    rms_v = float(torch.sqrt(torch.mean(qkv[2].float() ** 2)))
    assert np.abs(pick(out, rows) - sm).max() / rms_v <= 2e-2
    assert (its.numpy() <= w.cg_max_iters).all()
