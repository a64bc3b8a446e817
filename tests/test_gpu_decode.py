"""Decode step (one new query per (b, h) against a key/value cache) through the C ABI.

The step is row n-1 of the forward pass on the cached sequence, so the float64 oracle is the
LLA definition at that row.  Gates, per (b, h):
* CG run to convergence (relative residual 1e-6, fp32 arithmetic throughout): out within
  2^-8 |ref| + 1e-4 RMS(v) element by element (the first term covers the bf16 rounding of the
  output for bf16 caches; it is 0-width for fp32), rho within 2e-4 of RMS(ref rho), denom within
  2e-4 relative;
* at the LM configuration's fixed cap T = 16 the reference is the oracle's float64 run of the
  same centred CG for 16 iterations (truncation is part of the definition being compared), with
  the same bounds as the fp32 forward path at a fixed cap on converged rows.
Three forms compute the step (include/lla.h, lla_decode_ex): the moment form (tcgen05, the
default for bf16 caches at d = 128), and the streaming and cluster forms on CUDA cores.  Each
meets the same gates.
"""
import math

import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
from oracle.lla_ref import lla_row, lla_row_deflated_cg

pytestmark = pytest.mark.gpu
MOMENT, STREAM, CLUSTER = lla.LLA_DECODE_MOMENT, lla.LLA_DECODE_STREAM, lla.LLA_DECODE_CLUSTER
FORMS = {"moment": MOMENT, "stream": STREAM, "cluster": CLUSTER}


def _decode(w, n_cap=None, tol=None, iters=None, form=lla.LLA_DECODE_AUTO, inputs=None):
    q, k, v = make_inputs(w) if inputs is None else inputs   # [B, H, n, d]; the last row is the new token
    n = w.n
    n_cap = n if n_cap is None else n_cap
    dev = torch.device("cuda:0")
    kc = torch.zeros((w.B, w.H, n_cap, w.d), dtype=k.dtype)
    vc = torch.zeros_like(kc)
    kc[:, :, :n] = k
    vc[:, :, :n] = v
    if n_cap > n:                                # rows past n must not be read
        kc[:, :, n:] = float("nan")
        vc[:, :, n:] = float("nan")
    res = lla.decode(q[:, :, n - 1].contiguous().to(dev), kc.to(dev), vc.to(dev), n, w.tau, w.lam,
                     w.cg_max_iters if iters is None else iters, w.cg_tol if tol is None else tol, return_iters=True,
                     form=form)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return (q, k, v), [t.cpu() for t in res]


def _gate(w, qkv, res, ref_fn):
    q, k, v = (t.double().numpy() for t in qkv)
    out, rho, den, its = (t.double().numpy() for t in res)
    rms_v = math.sqrt(float(np.mean(v ** 2)))
    n = w.n
    for b in range(w.B):
        for h in range(w.H):
            r = ref_fn(q[b, h, n - 1], k[b, h, :n], v[b, h, :n])
            diff = np.abs(out[b, h] - r["out"])
            assert (diff <= 2.0 ** -8 * np.abs(r["out"]) * (w.dtype == "bf16") + 1e-4 * rms_v).all(), \
                f"out err {diff.max() / rms_v:.3e} RMS(v) at {(b, h)}"
            rms_rho = math.sqrt(float(np.mean(r["rho"] ** 2))) or 1.0
            assert np.abs(rho[b, h] - r["rho"]).max() <= 2e-4 * rms_rho
            assert abs(den[b, h] - r["denom"]) <= 2e-4 * abs(r["denom"])
    assert (its <= w.cg_max_iters).all()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("n", [1, 7, 33, 300])
def test_decode_converged_matches_exact_solve(lla_gpu, dtype, d, n):
    w = workload("lm_bf16", B=2, H=3, n=n, d=d, dtype=dtype, tau=1.0 / math.sqrt(d), cg_max_iters=4 * d + 64,
                 cg_tol=1e-6)
    qkv, res = _decode(w)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("dtype,n,B", [("bf16", 8000, 1), ("fp32", 4000, 1), ("bf16", 600, 50)])
def test_decode_streaming_form(lla_gpu, dtype, n, B):
    """The streaming form (K re-read every pass): for fp32 caches AUTO takes it for caches too long
    for an eighth to sit in a CTA's shared memory, and batches of more than 64 heads; the cluster
    form the rest.  At bf16 it is asked for by name."""
    w = workload("lm_bf16", B=B, H=3, n=n, d=128, dtype=dtype, tau=1.0 / math.sqrt(128), cg_max_iters=576,
                 cg_tol=1e-6)
    qkv, res = _decode(w, form=STREAM if dtype == "bf16" else lla.LLA_DECODE_AUTO)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("n", [1, 63, 64, 65, 129, 700])
def test_decode_moment_form_chunks_and_ragged_tail(lla_gpu, n):
    """The moment form over one key, one chunk of 64 keys, a chunk and one, and several chunks with
    a ragged last one (keys past n read as zeros and weighted 0)."""
    w = workload("lm_bf16", B=2, H=3, n=n, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=576, cg_tol=1e-6)
    qkv, res = _decode(w, form=MOMENT)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


def _rising_logits(w, step):
    """Inputs whose logits rise by about `step` per chunk of 64 keys: key j moves along the new
    query by (step * (j // 64)) / (tau |q|^2), so the weight sits on the last keys, which share a
    component along q many times their spread.  The caches hold the bf16 values."""
    q, k, v = make_inputs(w)
    qn = q[:, :, w.n - 1:w.n].double()
    shift = step * (torch.arange(w.n, dtype=torch.float64) // 64).view(1, 1, -1, 1)
    k = (k.double() + shift * qn / (w.tau * (qn * qn).sum(-1, keepdim=True))).to(k.dtype)
    return q, k, v


@pytest.mark.parametrize("form", ["moment", "stream"])
def test_decode_rising_maximum(lla_gpu, form):
    """Logits rising by ~3 per chunk over 11 chunks: every running maximum grows chunk after chunk,
    and the weighted keys share a large common component, which moments about any point but kbar
    would cancel at second order (the moment form centres on the exact kbar of its first pass).
    Same gate as every form."""
    w = workload("lm_bf16", B=2, H=3, n=700, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=576, cg_tol=1e-6)
    inputs = _rising_logits(w, 3.0)
    qkv, res = _decode(w, form=FORMS[form], inputs=inputs)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("B,n", [(80, 130), (160, 65)])
def test_decode_moment_form_many_heads_per_cta(lla_gpu, B, n):
    """More heads than SMs: each CTA takes two to five heads in turn, alternating its two TMEM
    accumulators and moment buffers (every head gated)."""
    w = workload("lm_bf16", B=B, H=4, n=n, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=576, cg_tol=1e-6)
    qkv, res = _decode(w, form=MOMENT)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
def test_decode_streaming_form_small_heads(lla_gpu, dtype, d):
    """The streaming form at every smaller head dimension (150 heads: past the cluster form's
    range), with a cache length that leaves a ragged last group of keys and a ragged last batch
    of the rows each thread fetches ahead."""
    w = workload("lm_bf16", B=50, H=3, n=299, d=d, dtype=dtype, tau=1.0 / math.sqrt(d), cg_max_iters=4 * d + 64,
                 cg_tol=1e-6)
    qkv, res = _decode(w)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("form,B", [("moment", 2), ("moment", 100), ("cluster", 2), ("stream", 75)])
def test_decode_reads_only_the_valid_cache_rows(lla_gpu, form, B):
    """n_cap > n: rows past n hold NaN and must not reach the result."""
    w = workload("lm_bf16", B=B, H=2, n=200, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=300, cg_tol=1e-6)
    qkv, res = _decode(w, n_cap=333, form=FORMS[form])
    assert all(np.isfinite(t.double().numpy()).all() for t in res[:3])
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))


@pytest.mark.parametrize("form", ["moment", "stream", "cluster"])
def test_decode_at_the_lm_cap_matches_the_same_cg(lla_gpu, form):
    """T = 16, tolerance 0 (the LM configuration): reference = float64 centred CG, 16 iterations."""
    w = workload("lm_bf16", B=2, H=4, n=2048, d=128)
    qkv, res = _decode(w, form=FORMS[form])
    q, k, v = (t.double().numpy() for t in qkv)
    out = res[0].double().numpy()
    rms_v = math.sqrt(float(np.mean(v ** 2)))
    n = w.n
    for b in range(w.B):
        for h in range(w.H):
            r = lla_row_deflated_cg(q[b, h, n - 1], k[b, h, :n], v[b, h, :n], w.tau, w.lam, 16, 0.0)
            diff = np.abs(out[b, h] - r["out"])
            assert (diff <= 2.0 ** -8 * np.abs(r["out"]) + 1e-3 * rms_v).all(), f"{diff.max() / rms_v:.3e}"
    assert (res[3].numpy() == 16).all()


def test_decode_full_size_sampled(lla_gpu):
    """The benchmark's decode configuration, in the launch the benchmark times (64 sequences x 16
    heads = 1024 heads: the moment form, about seven heads per CTA), against the float64 centred CG
    with the same cap T = 16 on sampled heads (first, last and six drawn with a fixed seed)."""
    w = workload("decode_bf16")
    q, k, v = make_inputs(w)
    n = w.n
    dev = torch.device("cuda:0")
    res = lla.decode(q[:, :, n - 1].contiguous().to(dev), k.to(dev), v.to(dev), n, w.tau, w.lam, w.cg_max_iters,
                     w.cg_tol, return_iters=True)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    out, rho, den, its = (t.cpu() for t in res)
    assert (its == w.cg_max_iters).all()
    assert torch.isfinite(out.float()).all() and torch.isfinite(rho).all() and (den > 0).all()
    rng = np.random.default_rng(11)
    heads = [(0, 0), (w.B - 1, w.H - 1)] + [(int(b), int(h)) for b, h in
                                             zip(rng.integers(0, w.B, 6), rng.integers(0, w.H, 6))]
    rms_v = math.sqrt(float(v[:2].double().pow(2).mean()))
    for b, h in heads:
        qi = q[b, h, n - 1].double().numpy()
        K, V = k[b, h].double().numpy(), v[b, h].double().numpy()
        r = lla_row_deflated_cg(qi, K, V, w.tau, w.lam, w.cg_max_iters, 0.0)
        diff = np.abs(out[b, h].double().numpy() - r["out"])
        assert (diff <= 2.0 ** -8 * np.abs(r["out"]) + 1e-3 * rms_v).all(), f"{(b, h)}: {diff.max() / rms_v:.3e}"


def test_decode_equals_forward_last_row(lla_gpu):
    """The step is the forward pass's row n-1: both fp32 GPU paths, same T, same inputs."""
    w = workload("lm_bf16", B=2, H=2, n=500, d=64, tau=0.125, cg_max_iters=200, cg_tol=1e-6)
    qkv, res = _decode(w)
    dev = torch.device("cuda:0")
    o, r, d_, _ = lla.forward(*(t.to(dev) for t in qkv), w.tau, w.lam, w.cg_max_iters, w.cg_tol,
                              path=lla.LLA_PATH_FP32, return_iters=True)
    torch.cuda.synchronize()
    rms_v = math.sqrt(float(qkv[2].double().pow(2).mean()))
    diff = (res[0].double() - o[:, :, -1].cpu().double()).abs()
    assert float(diff.max()) <= 2.0 ** -7 * float(o[:, :, -1].abs().max()) + 1e-4 * rms_v


def test_decode_moment_form_beyond_the_cuda_core_limit(lla_gpu):
    """A cache 1000 keys longer than the CUDA-core forms accept (they keep n weights in shared
    memory): AUTO takes the moment form, which keeps none.  out and rho meet the usual gate.  denom
    is held to 5e-4: the moment form's fp32 sums drift with n (denom measured 2e-5 relative at 4096
    keys, 1e-4 at 16384, 2.1e-4 at 32768 and 3.4e-4 here), which is why AUTO takes the CUDA-core
    forms between 16384 keys and their limit."""
    n = lla.lla_decode_max_n(128) + 1000
    w = workload("lm_bf16", B=1, H=2, n=n, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=576, cg_tol=1e-6)
    qkv, res = _decode(w)
    q, k, v = (t.double().numpy() for t in qkv)
    out, rho, den, _ = (t.double().numpy() for t in res)
    rms_v = math.sqrt(float(np.mean(v ** 2)))
    for h in range(w.H):
        r = lla_row(q[0, h, n - 1], k[0, h, :n], v[0, h, :n], w.tau, w.lam)
        assert (np.abs(out[0, h] - r["out"]) <= 2.0 ** -8 * np.abs(r["out"]) + 1e-4 * rms_v).all()
        assert np.abs(rho[0, h] - r["rho"]).max() <= 2e-4 * math.sqrt(float(np.mean(r["rho"] ** 2)))
        assert abs(den[0, h] - r["denom"]) <= 5e-4 * abs(r["denom"])
    with pytest.raises(lla.LLAError):
        _decode(w, form=STREAM)


def test_decode_auto_takes_a_cuda_core_form_between_16k_and_their_limit(lla_gpu):
    """At 32768 keys AUTO takes a CUDA-core form (the moment form's denom drifts to 2e-4 there),
    which meets the usual gate; the moment form, asked for by name, still serves the call."""
    w = workload("lm_bf16", B=1, H=2, n=32768, d=128, tau=1.0 / math.sqrt(128), cg_max_iters=576, cg_tol=1e-6)
    qkv, res = _decode(w)
    _gate(w, qkv, res, lambda qi, K, V: lla_row(qi, K, V, w.tau, w.lam))
    _, res_m = _decode(w, form=MOMENT)
    assert torch.isfinite(res_m[0].float()).all() and (res_m[2] > 0).all()
