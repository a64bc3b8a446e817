"""Causal Local Linear Attention (LLA) forward pass for GB300 (sm_103a).

Thin ctypes binding over liblla.so, whose C ABI is declared in include/lla.h.  The
binding only marshals arguments: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current stream.

There is no CPU fallback: if liblla.so is missing or cannot load, every call
raises ``LLAError``.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "LLAError", "load_library", "library_path", "forward", "forward_host", "lla_forward", "lla_forward_ex",
    "lla_forward_host", "lla_forward_host_buffer_size",
    "lla_workspace_size", "lla_resolve_path", "lla_sync_status", "lla_selftest_device_timeout", "lla_last_error",
    "lla_version",
    "lla_profile_enable", "lla_profile_read", "lla_forward_noalloc", "lla_parallax_forward", "parallax_forward",
    "lla_decode", "lla_decode_ex", "lla_decode_max_n", "decode", "lla_backward", "lla_backward_workspace_size", "backward",
    "lla_backward_host", "lla_backward_host_buffer_size", "backward_host",
    "LLA_OK", "LLA_ERR_INVALID_ARG", "LLA_ERR_UNSUPPORTED", "LLA_ERR_CUDA", "LLA_ERR_DEVICE_TIMEOUT",
    "LLA_DTYPE_BF16", "LLA_DTYPE_FP32", "LLA_PATH_AUTO", "LLA_PATH_TENSOR", "LLA_PATH_FP32",
    "LLA_DECODE_AUTO", "LLA_DECODE_MOMENT", "LLA_DECODE_STREAM", "LLA_DECODE_CLUSTER",
    "EXPORTED_SYMBOLS",
]

LLA_OK, LLA_ERR_INVALID_ARG, LLA_ERR_UNSUPPORTED, LLA_ERR_CUDA, LLA_ERR_DEVICE_TIMEOUT = range(5)
LLA_DTYPE_BF16, LLA_DTYPE_FP32 = 0, 1
LLA_PATH_AUTO, LLA_PATH_TENSOR, LLA_PATH_FP32 = 0, 1, 2
LLA_DECODE_AUTO, LLA_DECODE_MOMENT, LLA_DECODE_STREAM, LLA_DECODE_CLUSTER = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/lla.h
_SIGNATURES = {
    "lla_forward": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_float, _c_float,
                             _c_int, _c_float, _vp]),
    "lla_forward_ex": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                _c_float, _c_float, _c_int, _c_float, _vp, _c_size, _vp]),
    "lla_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "lla_forward_host": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                  _c_float, _c_float, _c_int, _c_float, _c_int, _vp, _c_size, _vp]),
    "lla_forward_host_buffer_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "lla_resolve_path": (_c_int, [_c_int, _c_int, _c_int]),
    "lla_sync_status": (_c_int, [_vp]),
    "lla_selftest_device_timeout": (_c_int, [_vp]),
    "lla_last_error": (ctypes.c_char_p, []),
    "lla_forward_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_float,
                                     _c_float, _c_int, _c_float, _vp]),
    "lla_parallax_forward": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                      _c_float, _vp, _c_size, _vp]),
    "lla_decode": (_c_int, [_c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                            _c_float, _c_float, _c_int, _c_float, _vp]),
    "lla_decode_ex": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                               _c_int, _c_float, _c_float, _c_int, _c_float, _vp]),
    "lla_decode_max_n": (_c_int, [_c_int]),
    "lla_backward": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                              _c_int, _c_int, _c_float, _c_float, _c_int, _c_float, _vp, _c_size, _vp]),
    "lla_backward_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "lla_backward_host": (_c_int, [_c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                   _c_int, _c_int, _c_float, _c_float, _c_int, _c_float, _c_int, _vp, _c_size, _vp]),
    "lla_backward_host_buffer_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "lla_profile_enable": (_c_int, [_c_int]),
    "lla_profile_read": (_c_int, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]),
    "lla_version": (_c_int, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)


class LLAError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"LLA status {status}: {message}")
        self.status = status


def library_path():
    return os.environ.get("LLA_LIBRARY", os.path.join(_HERE, "liblla.so"))


def load_library():
    """Load liblla.so (built by ``build.build()``); raises LLAError if it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise LLAError(-1, f"{path} not found: build it with local_linear_attention_flashlla_gb300.build.build()")
    try:
        lib = ctypes.CDLL(path)
    except OSError as e:
        raise LLAError(-1, f"cannot load {path}: {e}") from e
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status):
    if status != LLA_OK:
        raise LLAError(status, load_library().lla_last_error().decode(errors="replace"))


def lla_last_error():
    return load_library().lla_last_error().decode(errors="replace")


def lla_version():
    return load_library().lla_version()


def lla_resolve_path(dtype, path, d):
    return load_library().lla_resolve_path(dtype, path, d)


def lla_workspace_size(dtype, path, B, H, n, d):
    return load_library().lla_workspace_size(dtype, path, B, H, n, d)


def lla_profile_enable(on=True):
    """Record CUDA events around each later call's dominant kernel (measurement support)."""
    _check(load_library().lla_profile_enable(1 if on else 0))


def lla_profile_read():
    """(dominant-kernel ms, whole-call ms) of the most recent profiled call."""
    a, b = ctypes.c_float(), ctypes.c_float()
    _check(load_library().lla_profile_read(ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def lla_sync_status(stream=None):
    """Synchronise the stream and raise if a kernel recorded a device-side wait timeout."""
    _check(load_library().lla_sync_status(_stream_ptr(stream)))


def lla_selftest_device_timeout(stream=None):
    """Launch the library's timeout self-test kernel (a bounded wait that gives up after about two
    seconds); the next lla_sync_status(stream) raises LLAError with LLA_ERR_DEVICE_TIMEOUT."""
    _check(load_library().lla_selftest_device_timeout(_stream_ptr(stream)))


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def lla_forward(q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, B, H, n, d, tau, lam, cg_max_iters, cg_tol,
                stream_ptr):
    """Raw C entry point on device pointers (ints); raises LLAError on a non-zero status."""
    _check(load_library().lla_forward(q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, B, H, n, d, tau, lam,
                                      cg_max_iters, cg_tol, stream_ptr))


def lla_forward_noalloc(q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, B, H, n, d, tau, lam, cg_max_iters,
                        cg_tol, stream_ptr):
    """C entry point that uses the library's fixed device scratch instead of allocating."""
    _check(load_library().lla_forward_noalloc(q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, B, H, n, d, tau,
                                              lam, cg_max_iters, cg_tol, stream_ptr))


def lla_forward_ex(dtype, path, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B, H, n, d, tau, lam,
                   cg_max_iters, cg_tol, ws_ptr, ws_bytes, stream_ptr):
    """Raw C entry point with dtype/path/iteration-count/workspace arguments."""
    _check(load_library().lla_forward_ex(dtype, path, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr,
                                         B, H, n, d, tau, lam, cg_max_iters, cg_tol, ws_ptr, ws_bytes, stream_ptr))


def lla_forward_host(dtype, path, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B, H, n, d, tau, lam,
                     cg_max_iters, cg_tol, chunk_slices, buf_ptr, buf_bytes, stream_ptr):
    """Raw C entry point of the host-buffer forward (pointers are host addresses, buf_ptr a device one)."""
    _check(load_library().lla_forward_host(dtype, path, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr,
                                           B, H, n, d, tau, lam, cg_max_iters, cg_tol, chunk_slices, buf_ptr,
                                           buf_bytes, stream_ptr))


def lla_forward_host_buffer_size(dtype, path, B, H, n, d, chunk_slices=0):
    return load_library().lla_forward_host_buffer_size(dtype, path, B, H, n, d, chunk_slices)


def lla_parallax_forward(dtype, path, q_ptr, k_ptr, v_ptr, probe_ptr, out_ptr, B, H, n, d, tau, ws_ptr, ws_bytes,
                         stream_ptr):
    """Raw Parallax-form entry point on device pointers (ints); raises LLAError on failure."""
    _check(load_library().lla_parallax_forward(dtype, path, q_ptr, k_ptr, v_ptr, probe_ptr, out_ptr, B, H, n, d, tau,
                                               ws_ptr, ws_bytes, stream_ptr))


def lla_decode(dtype, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B, H, n, n_cap, d, tau, lam,
               cg_max_iters, cg_tol, stream_ptr):
    """Raw decode-step entry point on device pointers (ints); raises LLAError on failure."""
    _check(load_library().lla_decode(dtype, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B, H, n,
                                     n_cap, d, tau, lam, cg_max_iters, cg_tol, stream_ptr))


def lla_decode_ex(form, dtype, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B, H, n, n_cap, d, tau,
                  lam, cg_max_iters, cg_tol, stream_ptr):
    """Raw decode-step entry point with the form chosen (an LLA_DECODE_* value); raises LLAError."""
    _check(load_library().lla_decode_ex(form, dtype, q_ptr, k_ptr, v_ptr, out_ptr, rho_ptr, denom_ptr, iters_ptr, B,
                                        H, n, n_cap, d, tau, lam, cg_max_iters, cg_tol, stream_ptr))


def lla_decode_max_n(d):
    return load_library().lla_decode_max_n(d)


def decode(q, k_cache, v_cache, n, tau, lam, cg_max_iters, cg_tol=0.0, *, return_iters=False, out=None, rho=None,
           denom=None, form=LLA_DECODE_AUTO, stream=None):
    """One decode step: q [B, H, d] against caches [B, H, n_cap, d] whose first n rows are valid.

    Returns (out [B, H, d], rho [B, H, d] fp32, denom [B, H] fp32) and, with return_iters, the
    CG iteration counts [B, H].  Equals row n-1 of forward() on the cached sequence.  form: an
    LLA_DECODE_* value (include/lla.h, lla_decode_ex).
    """
    import torch
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda):
        raise LLAError(LLA_ERR_INVALID_ARG, "q and the caches must be CUDA tensors (there is no CPU path)")
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape or \
            tuple(k_cache.shape[:2]) != tuple(q.shape[:2]) or k_cache.shape[3] != q.shape[2]:
        raise LLAError(LLA_ERR_INVALID_ARG, f"q [B, H, d] and caches [B, H, n_cap, d] expected, got {tuple(q.shape)}, "
                                            f"{tuple(k_cache.shape)}, {tuple(v_cache.shape)}")
    if not (q.dtype == k_cache.dtype == v_cache.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise LLAError(LLA_ERR_INVALID_ARG, "q and the caches must all be bf16 or all fp32")
    q, k_cache, v_cache = q.contiguous(), k_cache.contiguous(), v_cache.contiguous()
    B, H, n_cap, d = k_cache.shape
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32
    if out is None:
        out = torch.empty_like(q)
    if rho is None:
        rho = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    if denom is None:
        denom = torch.empty((B, H), dtype=torch.float32, device=q.device)
    iters = torch.empty((B, H), dtype=torch.int32, device=q.device) if return_iters else None
    lla_decode_ex(int(form), dtype, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                  rho.data_ptr(), denom.data_ptr(), None if iters is None else iters.data_ptr(), B, H, int(n), n_cap, d,
                  float(tau), float(lam), int(cg_max_iters), float(cg_tol), _stream_ptr(stream))
    if return_iters:
        return out, rho, denom, iters
    return out, rho, denom


def lla_backward(dtype, path, q_ptr, k_ptr, v_ptr, rho_ptr, denom_ptr, dout_ptr, dq_ptr, dk_ptr, dv_ptr, iters_ptr,
                 B, H, n, d, tau, lam, cg_max_iters, cg_tol, ws_ptr, ws_bytes, stream_ptr):
    """Raw backward entry point on device pointers (ints); raises LLAError on failure."""
    _check(load_library().lla_backward(dtype, path, q_ptr, k_ptr, v_ptr, rho_ptr, denom_ptr, dout_ptr, dq_ptr, dk_ptr,
                                       dv_ptr, iters_ptr, B, H, n, d, tau, lam, cg_max_iters, cg_tol, ws_ptr,
                                       ws_bytes, stream_ptr))


def lla_backward_workspace_size(dtype, path, B, H, n, d):
    return load_library().lla_backward_workspace_size(dtype, path, B, H, n, d)


def backward(q, k, v, rho, denom, dout, tau, lam, cg_max_iters, cg_tol=0.0, *, path=LLA_PATH_AUTO,
             return_iters=False, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) [B, H, n, d] fp32 of sum(dout * out) for the forward call that gave
    rho [B, H, n, d] and denom [B, H, n] on q, k, v (see include/lla.h).  With return_iters also
    the adjoint CG iteration counts [B, H, n].  Asynchronous on the current (or given) stream.
    """
    import torch
    _check_qkv(q, k, v)
    if tuple(dout.shape) != tuple(q.shape) or dout.dtype != q.dtype or not dout.is_cuda:
        raise LLAError(LLA_ERR_INVALID_ARG, f"dout must be a CUDA tensor of shape {tuple(q.shape)} and dtype {q.dtype}")
    B, H, n, d = q.shape
    if tuple(rho.shape) != (B, H, n, d) or tuple(denom.shape) != (B, H, n) or \
            rho.dtype != torch.float32 or denom.dtype != torch.float32:
        raise LLAError(LLA_ERR_INVALID_ARG, "rho [B, H, n, d] and denom [B, H, n] must be the forward's fp32 outputs")
    q, k, v, dout = q.contiguous(), k.contiguous(), v.contiguous(), dout.contiguous()
    rho, denom = rho.contiguous(), denom.contiguous()
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32
    grads = []
    for t in (dq, dk, dv):
        grads.append(torch.empty((B, H, n, d), dtype=torch.float32, device=q.device) if t is None else t)
    iters = torch.empty((B, H, n), dtype=torch.int32, device=q.device) if return_iters else None
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    lla_backward(dtype, path, q.data_ptr(), k.data_ptr(), v.data_ptr(), rho.data_ptr(), denom.data_ptr(), dout.data_ptr(),
                 grads[0].data_ptr(), grads[1].data_ptr(), grads[2].data_ptr(),
                 None if iters is None else iters.data_ptr(), B, H, n, d, float(tau), float(lam), int(cg_max_iters),
                 float(cg_tol), ws_ptr, ws_bytes, _stream_ptr(stream))
    if return_iters:
        return (*grads, iters)
    return tuple(grads)


def lla_backward_host(dtype, path, q_ptr, k_ptr, v_ptr, rho_ptr, denom_ptr, dout_ptr, dq_ptr, dk_ptr, dv_ptr,
                      iters_ptr, B, H, n, d, tau, lam, cg_max_iters, cg_tol, chunk_slices, buf_ptr, buf_bytes,
                      stream_ptr):
    """Raw host-buffer backward entry point (host addresses; buf_ptr a device one)."""
    _check(load_library().lla_backward_host(dtype, path, q_ptr, k_ptr, v_ptr, rho_ptr, denom_ptr, dout_ptr, dq_ptr,
                                            dk_ptr, dv_ptr, iters_ptr, B, H, n, d, tau, lam, cg_max_iters, cg_tol,
                                            chunk_slices, buf_ptr, buf_bytes, stream_ptr))


def lla_backward_host_buffer_size(dtype, path, B, H, n, d, chunk_slices=0):
    return load_library().lla_backward_host_buffer_size(dtype, path, B, H, n, d, chunk_slices)


def backward_host(q, k, v, rho, denom, dout, tau, lam, cg_max_iters, cg_tol=0.0, *, path=LLA_PATH_AUTO,
                  chunk_slices=0, return_iters=False, dq=None, dk=None, dv=None, device_buffer=None, stream=None):
    """backward() on CPU tensors (pin them for overlapped copies): q, k, v, dout [B, H, n, d] bf16 or
    fp32, rho [B, H, n, d] and denom [B, H, n] fp32.  Returns CPU fp32 dq, dk, dv (pinned unless
    passed in).  Asynchronous on the current (or given) stream: synchronise before reading."""
    import torch
    ins = (q, k, v, dout, rho, denom)
    if any(t.is_cuda for t in ins):
        raise LLAError(LLA_ERR_INVALID_ARG, "backward_host takes CPU tensors; use backward() for CUDA tensors")
    if q.dim() != 4 or any(tuple(t.shape) != tuple(q.shape) for t in (k, v, dout, rho)):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v, dout, rho must share one [B, H, n, d] shape")
    B, H, n, d = q.shape
    if tuple(denom.shape) != (B, H, n) or rho.dtype != torch.float32 or denom.dtype != torch.float32:
        raise LLAError(LLA_ERR_INVALID_ARG, "rho [B, H, n, d] and denom [B, H, n] must be fp32")
    if not (q.dtype == k.dtype == v.dtype == dout.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v, dout must all be bf16 or all fp32")
    if not all(t.is_contiguous() for t in ins):
        raise LLAError(LLA_ERR_INVALID_ARG, "inputs must be contiguous (a copy would not stay alive for the call)")
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32
    grads = []
    for t in (dq, dk, dv):
        if t is None:
            t = torch.empty((B, H, n, d), dtype=torch.float32).pin_memory()
        elif t.is_cuda or tuple(t.shape) != (B, H, n, d) or t.dtype != torch.float32 or not t.is_contiguous():
            raise LLAError(LLA_ERR_INVALID_ARG, "gradient outputs must be contiguous CPU fp32 [B, H, n, d] tensors")
        grads.append(t)
    iters = torch.empty((B, H, n), dtype=torch.int32).pin_memory() if return_iters else None
    if device_buffer is None:
        buf_ptr, buf_bytes = None, 0
    else:
        if not device_buffer.is_cuda:
            raise LLAError(LLA_ERR_INVALID_ARG, "device_buffer must be a CUDA tensor")
        buf_ptr, buf_bytes = device_buffer.data_ptr(), device_buffer.numel() * device_buffer.element_size()
    lla_backward_host(dtype, path, q.data_ptr(), k.data_ptr(), v.data_ptr(), rho.data_ptr(), denom.data_ptr(),
                      dout.data_ptr(), grads[0].data_ptr(), grads[1].data_ptr(), grads[2].data_ptr(),
                      None if iters is None else iters.data_ptr(), B, H, n, d, float(tau), float(lam),
                      int(cg_max_iters), float(cg_tol), int(chunk_slices), buf_ptr, buf_bytes, _stream_ptr(stream))
    if return_iters:
        return (*grads, iters)
    return tuple(grads)


def _check_qkv(q, k, v):
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must be CUDA tensors (there is no CPU path)")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise LLAError(LLA_ERR_INVALID_ARG, f"q, k, v must share one [B, H, n, d] shape, got {tuple(q.shape)}, "
                                            f"{tuple(k.shape)}, {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must all be bf16 or all fp32")


def parallax_forward(q, k, v, probe, tau, *, path=LLA_PATH_AUTO, out=None, workspace=None, stream=None):
    """Parallax-form causal attention: softmax output minus Sigma_KV probe (see include/lla.h).

    q, k, v: CUDA [B, H, n, d] bf16 or fp32; probe: [B, H, n, d] (converted to contiguous fp32).
    Returns out (dtype of q).  Asynchronous on the current (or given) stream.
    """
    import torch
    _check_qkv(q, k, v)
    if tuple(probe.shape) != tuple(q.shape) or not probe.is_cuda:
        raise LLAError(LLA_ERR_INVALID_ARG, f"probe must be a CUDA tensor of shape {tuple(q.shape)}")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    probe = probe.to(torch.float32).contiguous()
    B, H, n, d = q.shape
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32
    if out is None:
        out = torch.empty_like(q)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    lla_parallax_forward(dtype, path, q.data_ptr(), k.data_ptr(), v.data_ptr(), probe.data_ptr(), out.data_ptr(),
                         B, H, n, d, float(tau), ws_ptr, ws_bytes, _stream_ptr(stream))
    return out


def forward(q, k, v, tau, lam, cg_max_iters, cg_tol=0.0, *, path=LLA_PATH_AUTO, return_iters=False,
            out=None, rho=None, denom=None, workspace=None, stream=None):
    """Causal LLA forward on CUDA tensors q, k, v of shape [B, H, n, d] (bf16 or fp32).

    Returns (out, rho, denom) or, with return_iters, (out, rho, denom, cg_iters).
    Output tensors are allocated with torch unless passed in.  Asynchronous on the
    current (or given) stream.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must be CUDA tensors (there is no CPU path)")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise LLAError(LLA_ERR_INVALID_ARG, f"q, k, v must share one [B, H, n, d] shape, got {tuple(q.shape)}, "
                                            f"{tuple(k.shape)}, {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must all be bf16 or all fp32")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, H, n, d = q.shape
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32
    if out is None:
        out = torch.empty_like(q)
    if rho is None:
        rho = torch.empty((B, H, n, d), dtype=torch.float32, device=q.device)
    if denom is None:
        denom = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    iters = torch.empty((B, H, n), dtype=torch.int32, device=q.device) if return_iters else None
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    lla_forward_ex(dtype, path, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), rho.data_ptr(),
                   denom.data_ptr(), None if iters is None else iters.data_ptr(), B, H, n, d, float(tau), float(lam),
                   int(cg_max_iters), float(cg_tol), ws_ptr, ws_bytes, _stream_ptr(stream))
    if return_iters:
        return out, rho, denom, iters
    return out, rho, denom


def forward_host(q, k, v, tau, lam, cg_max_iters, cg_tol=0.0, *, path=LLA_PATH_AUTO, chunk_slices=0,
                 return_iters=False, out=None, rho=None, denom=None, device_buffer=None, stream=None):
    """forward() on CPU tensors q, k, v [B, H, n, d] (bf16 or fp32; pin them for overlapped copies).

    The library copies the (b, h) slices to the GPU in chunks, computes and copies the results
    back into CPU tensors (pinned unless passed in), overlapping the transfers with the compute.
    Asynchronous on the current (or given) stream: synchronise it before reading the results.
    device_buffer: optional uint8 CUDA tensor of lla_forward_host_buffer_size(...) bytes.
    """
    import torch
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise LLAError(LLA_ERR_INVALID_ARG, "forward_host takes CPU tensors; use forward() for CUDA tensors")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise LLAError(LLA_ERR_INVALID_ARG, f"q, k, v must share one [B, H, n, d] shape, got {tuple(q.shape)}, "
                                            f"{tuple(k.shape)}, {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must all be bf16 or all fp32")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise LLAError(LLA_ERR_INVALID_ARG, "q, k, v must be contiguous (a copy would not stay alive for the call)")
    B, H, n, d = q.shape
    dtype = LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else LLA_DTYPE_FP32

    def host_out(t, shape, dt):
        if t is None:
            return torch.empty(shape, dtype=dt).pin_memory()
        if t.is_cuda or tuple(t.shape) != tuple(shape) or t.dtype != dt or not t.is_contiguous():
            raise LLAError(LLA_ERR_INVALID_ARG, f"output must be a contiguous CPU {dt} tensor of shape {tuple(shape)}")
        return t

    out = host_out(out, (B, H, n, d), q.dtype)
    rho = host_out(rho, (B, H, n, d), torch.float32)
    denom = host_out(denom, (B, H, n), torch.float32)
    iters = torch.empty((B, H, n), dtype=torch.int32).pin_memory() if return_iters else None
    if device_buffer is None:
        buf_ptr, buf_bytes = None, 0
    else:
        if not device_buffer.is_cuda:
            raise LLAError(LLA_ERR_INVALID_ARG, "device_buffer must be a CUDA tensor")
        buf_ptr, buf_bytes = device_buffer.data_ptr(), device_buffer.numel() * device_buffer.element_size()
    lla_forward_host(dtype, path, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), rho.data_ptr(),
                     denom.data_ptr(), None if iters is None else iters.data_ptr(), B, H, n, d, float(tau),
                     float(lam), int(cg_max_iters), float(cg_tol), int(chunk_slices), buf_ptr, buf_bytes,
                     _stream_ptr(stream))
    if return_iters:
        return out, rho, denom, iters
    return out, rho, denom
