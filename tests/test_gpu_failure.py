"""Failure detection on the GPU, without a fault.

The library's timeout self-test kernel waits, through the bounded and abortable mbarrier wait the
tensor kernels use, on a barrier that nothing arrives on.  The wait gives up after its limit
(about two seconds), the kernel records the timeout in the library's device error word and returns
normally.  These tests check the host side of that path, the boundary's documented error
behaviour: lla_sync_status reports LLA_ERR_DEVICE_TIMEOUT once and clears the word, and the CUDA
context and the library keep working afterwards.
"""
import time

import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import workload
from parity_util import run_gpu

pytestmark = pytest.mark.gpu


def test_device_timeout_is_reported_once(lla_gpu):
    lla.lla_sync_status()                          # nothing pending before the test
    t0 = time.monotonic()
    lla.lla_selftest_device_timeout()
    with pytest.raises(lla.LLAError) as ei:
        lla.lla_sync_status()
    elapsed = time.monotonic() - t0
    assert ei.value.status == lla.LLA_ERR_DEVICE_TIMEOUT
    assert "bounded device-side wait" in str(ei.value)
    # the wait ran to its limit (about 2 s) and no further
    assert 1.5 <= elapsed < 60.0, elapsed
    lla.lla_sync_status()                          # reported once: the word was cleared


def test_library_works_after_a_device_timeout(lla_gpu):
    """A tensor-path forward before and after the timeout gives bit-identical results (the
    forward's parity with the oracle is the tensor-path tests' subject)."""
    w = workload("lm_bf16", B=1, H=2, n=300, d=64, tau=0.125, cg_max_iters=200, cg_tol=1e-6)
    qkv, before = run_gpu(w, lla.LLA_PATH_TENSOR)
    lla.lla_selftest_device_timeout()
    with pytest.raises(lla.LLAError):
        lla.lla_sync_status()
    _, after = run_gpu(w, lla.LLA_PATH_TENSOR, inputs=qkv)
    for a, b in zip(before, after):
        assert torch.equal(a, b)
    out, rho, den, _ = after
    assert torch.isfinite(out.float()).all() and torch.isfinite(rho).all() and (den > 0).all()
