"""Every kernel maps its grid onto (query tile, head) pairs heaviest tile first, across groups of
heads whose operands fit in L2 together; the last group is ragged when the head count is not a
multiple of the group size.  The (b, h) slices are independent problems, so permuting the heads
of the inputs must permute the outputs bit for bit, and every output entry must be written.

Shapes: n = 4096 with d = 128 and 17 heads, or d = 64 and 33 heads.  The group sizes that gives
(32 MB of operands per group) are 16 + 1 (tensor forward, fp16 keys and values), 8 + 8 + 1 (fp32
forward), 10 + 7 and 16 + 1 (tensor backward: the query-side and key-side kernels) and
5 + 5 + 5 + 2 (fp32 backward) at d = 128, and ragged at d = 64 as well.  Outputs are prefilled
with NaN, so a (tile, head) pair that no CTA took stays visible.  Scales that the library takes
over the whole tensor (max |x| for the fp16 operands, per-key maxima) are the same under a
permutation of the heads, so the comparison is exact.
"""
import math

import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_cotangent, make_inputs, workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SHAPES = [(128, 17), (64, 33)]


def _inputs(d, H, dtype):
    w = workload("lm_bf16", B=1, H=H, n=4096, d=d, tau=1.0 / math.sqrt(d), dtype=dtype)
    q, k, v = (t.to(DEV) for t in make_inputs(w))
    perm = torch.randperm(H, generator=torch.Generator().manual_seed(7)).to(DEV)
    return w, (q, k, v), perm


def _nan(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device=DEV)


def _forward(w, q, k, v, path, tol):
    out = _nan(q.shape, q.dtype)
    rho = _nan(q.shape, torch.float32)
    den = _nan(q.shape[:3], torch.float32)
    lla.forward(q, k, v, w.tau, w.lam, w.cg_max_iters if tol == 0 else 96, tol, path=path,
                out=out, rho=rho, denom=den)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    return out, rho, den


def _check_permuted(a, b, perm, name):
    assert torch.isfinite(a.float()).all(), f"{name}: entries left unwritten or not finite"
    assert torch.equal(a[:, perm], b), f"{name}: permuting the heads changed the values"


@pytest.mark.parametrize("d,H", SHAPES)
@pytest.mark.parametrize("path,dtype,tol", [(lla.LLA_PATH_TENSOR, "bf16", 0.0),
                                            (lla.LLA_PATH_TENSOR, "bf16", 1e-5),
                                            (lla.LLA_PATH_FP32, "fp32", 0.0)],
                         ids=["tensor-cap", "tensor-tol", "fp32"])
def test_forward_head_permutation(lla_gpu, d, H, path, dtype, tol):
    w, (q, k, v), perm = _inputs(d, H, dtype)
    base = _forward(w, q, k, v, path, tol)
    moved = _forward(w, q[:, perm].contiguous(), k[:, perm].contiguous(), v[:, perm].contiguous(), path, tol)
    for a, b, name in zip(base, moved, ("out", "rho", "denom")):
        _check_permuted(a, b, perm, name)


@pytest.mark.parametrize("d,H", SHAPES)
@pytest.mark.parametrize("path,dtype", [(lla.LLA_PATH_TENSOR, "bf16"), (lla.LLA_PATH_FP32, "fp32")],
                         ids=["tensor", "fp32"])
def test_backward_head_permutation(lla_gpu, d, H, path, dtype):
    w, (q, k, v), perm = _inputs(d, H, dtype)
    _, rho, den = _forward(w, q, k, v, path, 0.0)
    g = make_cotangent(w).to(DEV)

    def run(*t):
        q_, k_, v_, rho_, den_, g_ = t
        grads = [_nan(q_.shape, torch.float32) for _ in range(3)]
        lla.backward(q_, k_, v_, rho_, den_, g_, w.tau, w.lam, w.cg_max_iters, 0.0, path=path,
                     dq=grads[0], dk=grads[1], dv=grads[2])
        torch.cuda.synchronize()
        lla.lla_sync_status()
        return grads

    base = run(q, k, v, rho, den, g)
    moved = run(*(t[:, perm].contiguous() for t in (q, k, v, rho, den, g)))
    for a, b, name in zip(base, moved, ("dq", "dk", "dv")):
        _check_permuted(a, b, perm, name)
