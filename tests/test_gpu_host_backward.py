"""The host-buffer backward (lla_backward_host): CPU tensors in and out, the (b, h) slices pushed
through the GPU in chunks on two library streams with the copies overlapped with the compute.

Each chunk's result is defined as lla_backward on that chunk's slices, so the checks are exact:
* fp32 path: bit-identical to one device backward over all slices;
* tensor path: bit-identical to device backwards over the same chunks, including a ragged last
  chunk, with the adjoint iteration counts returned.
The device backward's parity with the oracle is the subject of the backward tests.
"""
import math

import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_cotangent, make_inputs, workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(w):
    q, k, v = make_inputs(w)
    g = make_cotangent(w)
    o, rho, den = lla.forward(q.to(DEV), k.to(DEV), v.to(DEV), w.tau, w.lam, w.cg_max_iters, w.cg_tol)
    torch.cuda.synchronize()
    return [t.contiguous().pin_memory() for t in (q, k, v, g)] + [rho.cpu().pin_memory(), den.cpu().pin_memory()]


def _device(w, ins, path, sizes):
    q, k, v, g, rho, den = ins
    S = w.B * w.H
    flat = [t.reshape(S, 1, w.n, w.d) for t in (q, k, v, g, rho)] + [den.reshape(S, 1, w.n)]
    outs, s0 = [], 0
    for cnt in sizes:
        q_, k_, v_, g_, r_, d_ = (t[s0:s0 + cnt].to(DEV) for t in flat)
        s0 += cnt
        outs.append(lla.backward(q_, k_, v_, r_, d_, g_, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path,
                                 return_iters=True))
    torch.cuda.synchronize()
    shp = (w.B, w.H, w.n, w.d)
    cat = [torch.cat([o[i].cpu() for o in outs]) for i in range(4)]
    return cat[0].reshape(shp), cat[1].reshape(shp), cat[2].reshape(shp), cat[3].reshape(shp[:3])


def _host(w, ins, path, chunk):
    q, k, v, g, rho, den = ins
    res = lla.backward_host(q, k, v, rho, den, g, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path,
                            chunk_slices=chunk, return_iters=True)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return res


def _equal(a, b):
    for x, y in zip(a, b):
        assert x.shape == y.shape and x.dtype == y.dtype
        assert torch.equal(x, y)


@pytest.mark.parametrize("chunk", [0, 4])
def test_fp32_path_matches_one_device_call(lla_gpu, chunk):
    w = workload("lm_bf16", B=2, H=3, n=130, d=32, dtype="fp32", tau=1.0 / math.sqrt(32), cg_max_iters=40,
                 cg_tol=1e-6)
    ins = _inputs(w)
    _equal(_host(w, ins, lla.LLA_PATH_FP32, chunk), _device(w, ins, lla.LLA_PATH_FP32, [w.B * w.H]))


@pytest.mark.parametrize("d,chunk", [(64, 2), (128, 0)])
def test_tensor_path_matches_device_calls_per_chunk(lla_gpu, d, chunk):
    w = workload("lm_bf16", B=1, H=5, n=300, d=d)
    ins = _inputs(w)
    S = w.B * w.H
    C = chunk if chunk > 0 else (S + 7) // 8
    sizes = [min(C, S - s0) for s0 in range(0, S, C)]
    _equal(_host(w, ins, lla.LLA_PATH_TENSOR, chunk), _device(w, ins, lla.LLA_PATH_TENSOR, sizes))
