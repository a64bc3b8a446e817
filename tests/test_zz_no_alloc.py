"""The allocation-free entry point lla_forward_noalloc, through the C ABI.

It serves callers that cannot allocate device memory when they run the forward pass (their
memory belongs to another allocator, or the call must not pay for an allocation).  It must
give the same results as lla_forward on the same inputs, on consecutive calls that reuse its
fixed scratch, and must refuse problems larger than that scratch before launching anything.

This file is named to be collected last, and needs no state from other tests.
"""
import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload

pytestmark = pytest.mark.gpu


def _run(fn, w, q, k, v):
    out = torch.empty_like(q)
    rho = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    den = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), rho.data_ptr(), den.data_ptr(),
       w.B, w.H, w.n, w.d, w.tau, w.lam, w.cg_max_iters, w.cg_tol, stream)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return out.float(), rho, den


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_lla_forward_on_two_calls(lla_gpu, d):
    dev = torch.device("cuda:0")
    w = workload("lm_bf16", B=2, H=2, n=333, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=48)
    q, k, v = (t.to(dev) for t in make_inputs(w))
    ref_out, ref_rho, ref_den = _run(lla.lla_forward, w, q, k, v)
    rms_v = float(torch.sqrt(torch.mean(v.float() ** 2)))
    rms_rho = float(torch.sqrt(torch.mean(ref_rho ** 2)))
    # second problem in between so the second call finds the scratch holding other data
    w2 = workload("lm_bf16", B=1, H=3, n=200, d=d, tau=1.0 / np.sqrt(d), seed=7)
    q2, k2, v2 = (t.to(dev) for t in make_inputs(w2))
    for call in range(2):
        out, rho, den = _run(lla.lla_forward_noalloc, w, q, k, v)
        assert float((out - ref_out).abs().max()) / rms_v <= 2e-2, call
        assert float((rho - ref_rho).abs().max()) / rms_rho <= 2e-2, call
        assert float(((den - ref_den).abs() / ref_den.abs()).max()) <= 2e-2, call
        _run(lla.lla_forward_noalloc, w2, q2, k2, v2)


def test_noalloc_rejects_problems_beyond_its_scratch(lla_gpu):
    dev = torch.device("cuda:0")
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev)     # never read: rejected before launch
    f = torch.zeros(16, dtype=torch.float32, device=dev)
    lib = lla.load_library()
    # B*H*n*d large enough that the tensor path's scratch exceeds the fixed array
    st = lib.lla_forward_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), f.data_ptr(),
                                 f.data_ptr(), 8, 16, 4096, 128, 0.1, 1.0, 4, 0.0, None)
    assert st == lla.LLA_ERR_INVALID_ARG
    assert "scratch" in lla.lla_last_error()
    st = lib.lla_forward_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), f.data_ptr(),
                                 f.data_ptr(), 1, 1, 16, 32, 0.1, 1.0, 4, 0.0, None)
    assert st == lla.LLA_ERR_UNSUPPORTED
