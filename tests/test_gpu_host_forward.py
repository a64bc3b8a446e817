"""The host-buffer forward (lla_forward_host): CPU tensors in and out, the (b, h) slices pushed through
the GPU in chunks on two library streams with the copies overlapped with the compute.

Each chunk's result is defined as lla_forward_ex on that chunk's slices, so the checks are exact:
* fp32 path: bit-identical to one device forward over all slices (no per-call operand scaling);
* tensor path: bit-identical to device forwards over the same chunks (its fp16 operand scales are
  chosen per call), for several chunk sizes including a ragged last chunk;
* the same with a caller-supplied device buffer, with pageable (not pinned) host memory, and with
  the iteration counts returned.
The device forward's parity with the oracle is the subject of the tensor- and fp32-path tests.
"""
import math

import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload

pytestmark = pytest.mark.gpu


def _host_inputs(w, pinned=True):
    q, k, v = make_inputs(w)
    return tuple(t.contiguous().pin_memory() if pinned else t.contiguous() for t in (q, k, v))


def _device_chunks(w, q, k, v, path, chunk):
    """Device forwards over consecutive chunks of `chunk` (b, h) slices, as [S, 1, n, d] problems."""
    S = w.B * w.H
    dev = torch.device("cuda:0")
    flat = [t.reshape(S, 1, w.n, w.d) for t in (q, k, v)]
    outs = []
    for s0 in range(0, S, chunk):
        sl = [t[s0:s0 + chunk].to(dev) for t in flat]
        outs.append(lla.forward(*sl, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path, return_iters=True))
    torch.cuda.synchronize()
    cat = [torch.cat([o[i].cpu() for o in outs]) for i in range(4)]
    return (cat[0].reshape(q.shape), cat[1].reshape(w.B, w.H, w.n, w.d), cat[2].reshape(w.B, w.H, w.n),
            cat[3].reshape(w.B, w.H, w.n))


def _host(w, q, k, v, path, chunk, device_buffer=None):
    res = lla.forward_host(q, k, v, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path, chunk_slices=chunk,
                           return_iters=True, device_buffer=device_buffer)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return res


def _equal(a, b):
    for x, y in zip(a, b):
        assert x.shape == y.shape and x.dtype == y.dtype
        assert torch.equal(x, y)


@pytest.mark.parametrize("chunk", [0, 1, 4])
def test_fp32_path_matches_one_device_call(lla_gpu, chunk):
    w = workload("lm_bf16", B=2, H=3, n=130, d=32, dtype="fp32", tau=1.0 / math.sqrt(32), cg_max_iters=40,
                 cg_tol=1e-6)
    q, k, v = _host_inputs(w)
    dev = torch.device("cuda:0")
    ref = lla.forward(q.to(dev), k.to(dev), v.to(dev), w.tau, w.lam, w.cg_max_iters, w.cg_tol,
                      path=lla.LLA_PATH_FP32, return_iters=True)
    torch.cuda.synchronize()
    _equal(_host(w, q, k, v, lla.LLA_PATH_FP32, chunk), [t.cpu() for t in ref])


@pytest.mark.parametrize("chunk", [0, 2, 5])
def test_tensor_path_matches_device_calls_per_chunk(lla_gpu, chunk):
    w = workload("lm_bf16", B=1, H=5, n=300, d=64, tau=0.125, cg_max_iters=16, cg_tol=0.0)
    q, k, v = _host_inputs(w)
    S = w.B * w.H
    eff = chunk if chunk > 0 else (S + 7) // 8
    _equal(_host(w, q, k, v, lla.LLA_PATH_TENSOR, chunk), _device_chunks(w, q, k, v, lla.LLA_PATH_TENSOR, eff))


def test_tensor_path_lm_heads_with_a_caller_buffer_and_pageable_memory(lla_gpu):
    """d = 128, two sequences of 16 heads in chunks of 4 slices (8 chunks, both streams busy), the
    device buffer from the caller; then the same inputs from pageable memory."""
    w = workload("lm_bf16", B=2, H=16, n=257, d=128)
    q, k, v = _host_inputs(w)
    ref = _device_chunks(w, q, k, v, lla.LLA_PATH_TENSOR, 4)
    nbytes = lla.lla_forward_host_buffer_size(lla.LLA_DTYPE_BF16, lla.LLA_PATH_TENSOR, w.B, w.H, w.n, w.d, 4)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    _equal(_host(w, q, k, v, lla.LLA_PATH_TENSOR, 4, device_buffer=buf), ref)
    qp, kp, vp = _host_inputs(w, pinned=False)
    _equal(_host(w, qp, kp, vp, lla.LLA_PATH_TENSOR, 4), ref)


def test_small_device_buffer_is_rejected(lla_gpu):
    w = workload("lm_bf16", B=1, H=2, n=64, d=64)
    q, k, v = _host_inputs(w)
    buf = torch.empty(1024, dtype=torch.uint8, device="cuda:0")
    with pytest.raises(lla.LLAError) as ei:
        lla.forward_host(q, k, v, w.tau, w.lam, w.cg_max_iters, device_buffer=buf)
    assert ei.value.status == lla.LLA_ERR_INVALID_ARG
