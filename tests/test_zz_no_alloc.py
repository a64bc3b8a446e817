"""The allocation-free entry point lla_forward_noalloc, through the C ABI.

It serves callers that cannot allocate device memory when they run the forward pass (their
memory belongs to another allocator, or the call must not pay for an allocation).  It runs the
same tensor-path kernels as lla_forward on the same inputs, so its results must be bit-identical
to lla_forward's, on consecutive calls that reuse its fixed scratch with another problem in
between; it must allocate nothing from the device's stream-ordered pool; and it must refuse
problems larger than that scratch before launching anything.

This file is named to be collected last, and needs no state from other tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
from oracle.lla_ref import lla_ref

pytestmark = pytest.mark.gpu

LIMIT = 32 * 1024 * 1024          # LLA_NOALLOC_SCRATCH_BYTES in include/lla.h


def _run(name, w, q, k, v):
    """Call the C entry point `name` (lla_forward or lla_forward_noalloc) and wait for it."""
    fn = getattr(lla.load_library(), name)
    out = torch.empty_like(q)
    rho = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    den = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), rho.data_ptr(), den.data_ptr(),
            w.B, w.H, w.n, w.d, w.tau, w.lam, w.cg_max_iters, w.cg_tol, stream)
    torch.cuda.synchronize()
    assert st == lla.LLA_OK, lla.lla_last_error()
    lla.lla_sync_status()
    return out, rho, den


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


class _DevicePool:
    """Used-memory figures of the device's current stream-ordered pool (the pool cudaMallocAsync
    draws from), read through the CUDA driver API."""
    RESERVED_MEM_CURRENT, USED_MEM_CURRENT, USED_MEM_HIGH = 5, 7, 8   # CUmemPool_attribute

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        val = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(val)) == 0
        return val.value

    def reset_high(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_matches_lla_forward_on_two_calls(lla_gpu, d):
    dev = torch.device("cuda:0")
    w = workload("lm_bf16", B=2, H=2, n=333, d=d, tau=1.0 / np.sqrt(d), cg_max_iters=48)
    q, k, v = (t.to(dev) for t in make_inputs(w))
    ref = _run("lla_forward", w, q, k, v)
    # a second problem in between, so the second call finds the scratch holding other data
    w2 = workload("lm_bf16", B=1, H=3, n=200, d=d, tau=1.0 / np.sqrt(d), seed=7)
    q2, k2, v2 = (t.to(dev) for t in make_inputs(w2))
    for call in range(2):
        got = _run("lla_forward_noalloc", w, q, k, v)
        for name, a, b in zip(("out", "rho", "denom"), got, ref):
            assert _same_bits(a, b), f"call {call}: {name} differs from lla_forward"
        _run("lla_forward_noalloc", w2, q2, k2, v2)
    # and a few rows against the float64 oracle (CG at cap 48 has converged on this shape)
    rows = [(0, 0, 0), (0, 1, 127), (1, 0, 128), (1, 1, 332)]
    qn, kn, vn = (t.double().cpu().numpy() for t in (q, k, v))
    r_out = lla_ref(qn, kn, vn, w.tau, w.lam, rows=rows)[0]
    rms_v = math.sqrt(float(np.mean(vn ** 2)))
    g_out = np.array([got[0][b, h, i].double().cpu().numpy() for b, h, i in rows])
    assert np.abs(g_out - r_out).max() / rms_v <= 2e-2


def test_noalloc_allocates_nothing(lla_gpu):
    """Two calls leave the device pool's used and reserved bytes, and its high-water mark of
    used bytes, where they were; torch's allocator is not touched either."""
    dev = torch.device("cuda:0")
    w = workload("lm_bf16", B=1, H=2, n=300)
    q, k, v = (t.to(dev) for t in make_inputs(w))
    outs = [torch.empty_like(q), torch.empty(q.shape, dtype=torch.float32, device=dev),
            torch.empty(q.shape[:3], dtype=torch.float32, device=dev)]
    stream = torch.cuda.current_stream().cuda_stream
    lib = lla.load_library()

    def call():
        st = lib.lla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), *(t.data_ptr() for t in outs),
                                     w.B, w.H, w.n, w.d, w.tau, w.lam, w.cg_max_iters, w.cg_tol, stream)
        assert st == lla.LLA_OK, lla.lla_last_error()

    call()                        # first call on the device: any one-time module loading happens here
    torch.cuda.synchronize()
    pool = _DevicePool()
    used0, res0 = pool.get(pool.USED_MEM_CURRENT), pool.get(pool.RESERVED_MEM_CURRENT)
    torch_alloc0 = torch.cuda.memory_allocated()
    pool.reset_high()
    call()
    call()
    torch.cuda.synchronize()
    lla.lla_sync_status()
    assert pool.get(pool.USED_MEM_HIGH) == 0, "the call drew from the stream-ordered pool"
    assert pool.get(pool.USED_MEM_CURRENT) == used0
    assert pool.get(pool.RESERVED_MEM_CURRENT) == res0
    assert torch.cuda.memory_allocated() == torch_alloc0


def _largest_n_within(B, H, d):
    lo, hi = 1, 1
    while lla.lla_workspace_size(lla.LLA_DTYPE_BF16, lla.LLA_PATH_TENSOR, B, H, hi, d) <= LIMIT:
        lo, hi = hi, hi * 2
    while hi - lo > 1:        # largest n whose scratch fits: size(lo) <= LIMIT < size(hi)
        mid = (lo + hi) // 2
        if lla.lla_workspace_size(lla.LLA_DTYPE_BF16, lla.LLA_PATH_TENSOR, B, H, mid, d) <= LIMIT:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_at_its_size_limit(lla_gpu):
    """The largest problem that fits (a ragged last tile) runs and matches lla_forward bit for
    bit; one more row is rejected before launch."""
    d = 128
    B, n = next((B, n) for B in (1, 2, 3, 5, 7) for n in [_largest_n_within(B, 1, d)] if n % 128)
    assert lla.lla_workspace_size(lla.LLA_DTYPE_BF16, lla.LLA_PATH_TENSOR, B, 1, n, d) <= LIMIT
    dev = torch.device("cuda:0")
    w = workload("lm_bf16", B=B, H=1, n=n, cg_max_iters=4)
    q, k, v = (t.to(dev) for t in make_inputs(w))
    got = _run("lla_forward_noalloc", w, q, k, v)
    ref = _run("lla_forward", w, q, k, v)
    for name, a, b in zip(("out", "rho", "denom"), got, ref):
        assert _same_bits(a, b), f"{name} differs from lla_forward at n = {n}"
    assert torch.isfinite(got[0].float()).all() and (got[2] > 0).all()

    lib = lla.load_library()
    st = lib.lla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), *(t.data_ptr() for t in got),
                                 B, 1, n + 1, d, w.tau, w.lam, 4, 0.0, None)
    assert st == lla.LLA_ERR_INVALID_ARG
    assert "scratch" in lla.lla_last_error()


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
