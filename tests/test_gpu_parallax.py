"""Parallax-form forward (caller-supplied probe) through the C ABI, against the float64 oracle
(softmax output minus the explicitly formed softmax-weighted Sigma_KV times the probe).

Tolerances, element by element:
* fp32 path: |out - ref| <= 1e-4 RMS(v), the fp32 accumulation bound of the fp32 configurations;
* tensor path: |out - ref| <= 2^-8 |ref| + 2e-3 RMS(v).  There is no iterative solve here, so
  the error is rounding: the bf16 output itself (half an ulp, 2^-9 relative; 2^-8 leaves room
  for the value it rounds to be slightly off), plus fp16 per-pair coefficients (2^-11 relative
  each, averaged over the keys), the probe split into two fp16 halves (about 2^-22) and fp32
  accumulation, together well under 2e-3 of RMS(v) for these inputs.
"""
import math

import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, make_probe, workload
from oracle.lla_ref import parallax_ref, softmax_ref

pytestmark = pytest.mark.gpu


def _run(w, path, probe=None):
    q, k, v = make_inputs(w)
    r = make_probe(w) if probe is None else probe
    dev = torch.device("cuda:0")
    out = lla.parallax_forward(q.to(dev), k.to(dev), v.to(dev), r.to(dev), w.tau, path=path)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return (q, k, v, r), out.cpu()


def _err(w, qkvr, out, rows=None):
    """Per-row max of |out - ref| / RMS(v), and per-row max of the excess over the tensor-path
    bound 2^-8 |ref| + 2e-3 RMS(v) (<= 0 where the bound holds)."""
    q, k, v, r = (t.double().numpy() for t in qkvr)
    ref = parallax_ref(q, k, v, r, w.tau, rows=rows)
    got = out.double().numpy().reshape(-1, w.d) if rows is None else \
        np.array([out[b, h, i].double().numpy() for b, h, i in rows])
    rms_v = math.sqrt(float(np.mean(v ** 2)))
    diff = np.abs(got - ref)
    return diff.max(axis=1) / rms_v, (diff - (2.0 ** -8 * np.abs(ref) + 2e-3 * rms_v)).max(axis=1)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("n", [1, 33, 200])
def test_parallax_fp32_path(lla_gpu, d, n):
    w = workload("tiny_fp32", B=2, H=2, n=n, d=d, tau=1.0 / math.sqrt(d))
    qkvr, out = _run(w, lla.LLA_PATH_FP32)
    assert _err(w, qkvr, out)[0].max() <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 333])
def test_parallax_tensor_path(lla_gpu, d, n):
    w = workload("lm_bf16", B=2, H=2, n=n, d=d, tau=1.0 / math.sqrt(d))
    qkvr, out = _run(w, lla.LLA_PATH_TENSOR)
    e, excess = _err(w, qkvr, out)
    assert np.isfinite(out.float().numpy()).all()
    assert excess.max() <= 0.0, f"worst |err|/RMS(v) {e.max():.3e}, excess {excess.max():.3e}"


def test_parallax_zero_probe_is_softmax_on_gpu(lla_gpu):
    w = workload("lm_bf16", B=1, H=2, n=300, d=128, tau=1.0 / math.sqrt(128))
    zero = torch.zeros((w.B, w.H, w.n, w.d))
    qkvr, out = _run(w, lla.LLA_PATH_TENSOR, probe=zero)
    q, k, v = (t.double().numpy() for t in qkvr[:3])
    ref = softmax_ref(q, k, v, w.tau)
    rms_v = math.sqrt(float(np.mean(v ** 2)))
    diff = np.abs(out.double().numpy().reshape(-1, w.d) - ref)
    assert (diff <= 2.0 ** -8 * np.abs(ref) + 2e-3 * rms_v).all()


def test_parallax_full_size_sampled(lla_gpu):
    """LM-shaped workload at full size (B=8, H=16, n=4096, d=128): sampled rows."""
    from local_linear_attention_flashlla_gb300.inputs import sample_rows
    w = workload("lm_bf16")
    qkvr, out = _run(w, lla.LLA_PATH_AUTO)
    rows = sample_rows(w, 96)
    e, excess = _err(w, qkvr, out, rows=rows)
    assert excess.max() <= 0.0, f"worst |err|/RMS(v) {e.max():.3e}, excess {excess.max():.3e}"


@pytest.mark.parametrize("d", [64, 128])
def test_parallax_tensor_path_row_maximum_far_past_the_first_block(lla_gpu, d):
    """Keys 128..255 scaled by 4: rows past the first tile have their maximum far above the first key
    block's (the tiles the launch without a MAX sweep marks for the second launch).  Same bound."""
    w = workload("lm_bf16", B=1, H=2, n=300, d=d, tau=1.0 / math.sqrt(d))
    q, k, v = (t.clone() for t in make_inputs(w))
    k[:, :, 128:256] = (k[:, :, 128:256].float() * 4.0).bfloat16()
    r = make_probe(w)
    dev = torch.device("cuda:0")
    out = lla.parallax_forward(q.to(dev), k.to(dev), v.to(dev), r.to(dev), w.tau, path=lla.LLA_PATH_TENSOR)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    _, excess = _err(w, (q, k, v, r), out.cpu())
    assert excess.max() <= 0.0, float(excess.max())
